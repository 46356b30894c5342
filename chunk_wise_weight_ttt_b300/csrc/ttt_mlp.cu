// Host side of the C ABI declared in include/ttt_mlp.h: argument checks,
// workspace carving, chunk/group planning, tensor-map encoding and kernel
// launches for the two kernel families (tcgen05 bf16 path, fp32 SIMT path).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ttt_mlp.h"
#include "simt_kernels.cuh"
#include "tc_gemm.cuh"

using namespace ttt;

struct ttt_mlp {
  ttt_mlp_config cfg;
  const void *wg, *wu, *w0, *conv, *wt;
  bool tc;
  int G, L, s_pad, s_slots, num_sms;
  int max_pairs;            // co-resident CTA pairs of the tcgen05 kernels
  float* W;                 // fp32 path: n_docs x d x f
  uint16_t* Whi;            // tcgen05 path: n_docs x 2 x d x f hi planes of the fp32 state
  uint16_t* Wlo;            // tcgen05 path: n_docs x d x f lo planes
  __nv_bfloat16* WtT;       // W_target transposed (out x in)
  void *Z, *U, *V;          // per-call intermediates (n x f, n x d, n x d)
  __nv_bfloat16* S;         // s_slots blocks of s_pad x s_pad
  float *GZ, *GV;           // same-chunk Gram blocks for update clipping (or null)
  void *xs, *x0s, *os;      // host-staging copies of x, x0, o
  // A handle that owns its scratch has two staging buffers for x and x0 and
  // alternates them between host-buffer calls, so that a call's input copies
  // can run while the previous call's layers do.
  bool owns_scratch = false;
  void *xs2 = nullptr, *x0s2 = nullptr;
  int stage_sel = 0;
  cudaEvent_t ev_free[2] = {nullptr, nullptr};  // the layers that read staging buffer b are done
  int* ctrl;                // [0] error word, [64..] tile counters
  int counter_next;
  std::vector<uint8_t> hcur;  // per slot: which of its two hi planes is current
  CUtensorMap map_wg, map_wu, map_wtT, map_s, map_w0;
  std::string err;
  // benchmark phase timing
  bool profiling;
  struct Rec {
    int phase;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  int64_t prof_calls, prof_group_launches, prof_launches;
  // host-buffer calls: the copy streams and events of the segment pipeline
  // (created on first use)
  cudaStream_t st_in = nullptr, st_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in = nullptr, ev_out = nullptr;
  ~ttt_mlp() {
    for (cudaEvent_t e : {ev_start, ev_in, ev_out, ev_free[0], ev_free[1]})
      if (e) cudaEventDestroy(e);
    for (cudaStream_t q : {st_in, st_out})
      if (q) cudaStreamDestroy(q);
  }
};

namespace {

thread_local std::string g_err;

constexpr int kCtrlInts = 4096;
constexpr int kCounterBase = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool fault_injected(const char* name) {
  const char* f = std::getenv("TTT_FAULT");
  return f && std::strcmp(f, name) == 0;
}

bool force_simt() {
  const char* f = std::getenv("TTT_FORCE_SIMT");
  return f && f[0] == '1';
}

// Tokens per group of the tcgen05 path.  The fast weight is streamed through
// HBM once per group while the intra-group correction (Gram blocks) grows with
// the group; on a B300 at the Qwen3-4B layer shape 2048 measured best (group
// kernel 75% of the sustained bf16 peak; 1024: 64%, 512: 46%; whole layer
// +3% over 1024).  The TTT_GROUP_TOKENS environment variable (256..4096) is a
// tuning override.
int group_tokens() {
  static const int g = [] {
    const char* v = std::getenv("TTT_GROUP_TOKENS");
    const int n = v ? std::atoi(v) : 2048;
    return (n >= 256 && n <= 4096) ? n : 2048;
  }();
  return g;
}

// Workspace layout.  The state part (control block, fast weights, their bf16
// operand copies, the transposed W_target) belongs to one handle; the scratch
// part (per-call intermediates and host staging) may be shared by handles
// whose calls are ordered one after another.  Offsets of each part are
// relative to that part's base.
struct Layout {
  bool tc;
  int G, L, s_pad, s_slots;
  size_t ctrl, W, Whi, Wlo, WtT, state_total;               // state part
  size_t Z, U, V, S, GZ, GV, xs, x0s, os, xs2, x0s2, scratch_total;  // scratch part
};

bool config_ok(const ttt_mlp_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("config is NULL");
  if (c->d < 8 || c->d % 8) return bad("d must be a positive multiple of 8");
  if (c->f < 8 || c->f % 8) return bad("f must be a positive multiple of 8");
  if (c->chunk < 1 || c->chunk > 1024) return bad("chunk must be in 1..1024");
  if (c->conv_k < 1 || c->conv_k > 8) return bad("conv_k must be in 1..8");
  if (c->n_docs < 1 || c->n_docs > 4096) return bad("n_docs must be in 1..4096");
  if (c->act_dtype != TTT_F32 && c->act_dtype != TTT_BF16) return bad("act_dtype must be TTT_F32 or TTT_BF16");
  if (c->max_tokens < 1 || c->max_tokens > (int64_t(1) << 24)) return bad("max_tokens must be in 1..2^24");
  if (!std::isfinite(c->eta)) return bad("eta must be finite");
  if (c->target_mode < TTT_TARGET_NEXT || c->target_mode > TTT_TARGET_CAUSAL)
    return bad("target_mode must be TTT_TARGET_NEXT, TTT_TARGET_CURRENT or TTT_TARGET_CAUSAL");
  if (!std::isfinite(c->clip_tau) || c->clip_tau < 0.0f) return bad("clip_tau must be 0 (off) or a positive finite number");
  return true;
}

bool tc_shape_ok(const ttt_mlp_config& c) {
  return c.act_dtype == TTT_BF16 && c.d % 64 == 0 && c.f % 64 == 0 && c.d >= 256 && c.f >= 256;
}

Layout make_layout(const ttt_mlp_config& c, bool tc) {
  Layout l{};
  l.tc = tc;
  const size_t act = (c.act_dtype == TTT_BF16) ? 2 : 4;
  const size_t inter = tc ? 2 : 4;
  const size_t d = c.d, f = c.f, n = (size_t)c.max_tokens;
  l.G = tc ? std::max(1, group_tokens() / c.chunk) : 1;
  l.L = l.G * c.chunk;
  l.s_pad = (int)align_up((size_t)l.L, 256);
  l.s_slots = tc ? (int)std::min<int64_t>(kMaxGroups, (c.max_tokens + l.L - 1) / l.L + 4) : 0;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  l.ctrl = take(kCtrlInts * sizeof(int));
  // the fp32 state: fp32 values on the fp32 path; two hi planes and a lo
  // plane (16 bits each) per slot on the tcgen05 path
  l.W = tc ? 0 : take((size_t)c.n_docs * d * f * 4);
  l.Whi = tc ? take((size_t)c.n_docs * 2 * d * f * 2) : 0;
  l.Wlo = tc ? take((size_t)c.n_docs * d * f * 2) : 0;
  l.WtT = tc ? take(d * d * 2) : 0;
  l.state_total = o;
  o = 0;
  l.Z = take(n * f * inter);
  l.U = take(n * d * inter);
  l.V = take(n * d * inter);
  l.S = tc ? take((size_t)l.s_slots * l.s_pad * l.s_pad * 2) : 0;
  // same-chunk Gram blocks of Z and V for update clipping (fp32): per group
  // of a wave on the tcgen05 path, one chunk at a time on the fp32 path
  const size_t gram = c.clip_tau > 0.0f
                          ? (tc ? (size_t)l.s_slots * l.s_pad * l.s_pad : (size_t)c.chunk * c.chunk) * 4
                          : 0;
  l.GZ = gram ? take(gram) : 0;
  l.GV = gram ? take(gram) : 0;
  l.xs = take(n * d * act);
  l.x0s = take(n * d * act);
  l.os = take(n * d * act);
  l.xs2 = take(n * d * act);
  l.x0s2 = take(n * d * act);
  l.scratch_total = o;
  return l;
}

// Bytes of each part the handle may need: the larger of the two kernel
// families' layouts (which family runs is decided at create).
size_t state_bytes_of(const ttt_mlp_config& c) {
  size_t b = make_layout(c, false).state_total;
  if (tc_shape_ok(c)) b = std::max(b, make_layout(c, true).state_total);
  return b;
}
size_t scratch_bytes_of(const ttt_mlp_config& c) {
  size_t b = make_layout(c, false).scratch_total;
  if (tc_shape_ok(c)) b = std::max(b, make_layout(c, true).scratch_total);
  return b;
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Matrix [outer x inner] row-major with row pitch `pitch` elements (bf16, or
// fp32 when `f32`); box (box_inner x box_outer) with 128-byte swizzle, zero
// fill outside.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
              uint32_t box_inner, uint32_t box_outer, std::string* why, bool f32 = false) {
  auto fn = encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is unavailable";
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu map",
                  (int)r, (unsigned long long)outer, (unsigned long long)inner);
    *why = buf;
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- errors

ttt_status fail(ttt_mlp* h, ttt_status s, const std::string& msg) {
  if (h)
    h->err = msg;
  else
    g_err = msg;
  return s;
}

#define TTT_CK(h, expr)                                                                    \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return fail((h), TTT_ECUDA, std::string(#expr) + ": " + cudaGetErrorString(e_));     \
  } while (0)

#define TTT_CK_LAUNCH(h) TTT_CK(h, cudaGetLastError())

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch shape of conv_target_kernel<TIn, ., .> for the tokens the span list covers.
template <typename TIn>
dim3 conv_grid(const SpanList& sl, int d) {
  const int ntok = sl.start[sl.n - 1] + sl.len[sl.n - 1] - sl.start[0];
  constexpr int tok = conv_tokens<TIn>();
  return dim3((unsigned)((ntok + tok - 1) / tok), (unsigned)((d + kConvCh - 1) / kConvCh));
}

int grid_for(long long n, int block) {
  long long g = (n + block - 1) / block;
  return (int)std::max<long long>(1, std::min<long long>(g, 1 << 20));
}

// ---------------------------------------------------------------- planning

struct Span {
  int start, len;
  bool reset;
};

// Chunks of one call (a document start restarts the chunking; the call starts
// a fresh chunk at token 0), then groups of up to G consecutive chunks of one
// document.  Only a group's last chunk can be shorter than C.
std::vector<Span> plan_groups(int64_t n, int C, int G, const int64_t* ds, int nds) {
  std::vector<int64_t> cuts;
  cuts.push_back(0);
  for (int i = 0; i < nds; ++i)
    if (ds[i] > 0) cuts.push_back(ds[i]);
  cuts.push_back(n);
  std::vector<Span> out;
  for (size_t i = 0; i + 1 < cuts.size(); ++i) {
    const int64_t a = cuts[i], b = cuts[i + 1];
    const bool doc = (i > 0) || (nds > 0 && ds[0] == 0);
    for (int64_t t = a; t < b; t += (int64_t)G * C) {
      const int64_t e = std::min<int64_t>(t + (int64_t)G * C, b);
      out.push_back(Span{(int)t, (int)(e - t), doc && t == a});
    }
  }
  return out;
}

int cdiv_h(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch of the tcgen05 kernels (on unless TTT_PDL=0).
bool use_pdl() {
  static const bool on = [] {
    const char* v = std::getenv("TTT_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Launch the tcgen05 engine as clusters of two CTAs: one persistent cluster
// per co-resident CTA pair, at most one per tile pair.  With programmatic
// dependent launch the grid's prologue overlaps the previous kernel's tail;
// the kernel waits for that kernel before it touches global memory.
template <int MODE>
cudaError_t launch_pairs(int max_pairs, const GemmArgs& a, int npairs, cudaStream_t st) {
  if (npairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2 * std::max(1, std::min(max_pairs, npairs)));
  lc.blockDim = dim3(kGemmThreads);
  lc.dynamicSmemBytes = smem_bytes_of<MODE>();
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = use_pdl() ? 2 : 1;
  return cudaLaunchKernelEx(&lc, tc_gemm_kernel<MODE>, a);
}

template <int MODE>
cudaError_t launch_gemm(ttt_mlp* h, GemmArgs& a, int npairs, cudaStream_t st) {
  return launch_pairs<MODE>(h->max_pairs, a, npairs, st);
}

// Kernel attributes of the tcgen05 engine and the number of CTA pairs that can
// be resident at once (0 on failure).
cudaError_t setup_tc_kernels(int* max_pairs) {
  const void* kfn[5] = {(const void*)tc_gemm_kernel<kSwiGLU>, (const void*)tc_gemm_kernel<kLinear>,
                        (const void*)tc_gemm_kernel<kSGram>, (const void*)tc_gemm_kernel<kGroup>,
                        (const void*)tc_gemm_kernel<kDGram>};
  const int smem[5] = {smem_bytes_of<kSwiGLU>(), smem_bytes_of<kLinear>(), smem_bytes_of<kSGram>(),
                       smem_bytes_of<kGroup>(), smem_bytes_of<kDGram>()};
  for (int i = 0; i < 5; ++i) {
    cudaError_t e = cudaFuncSetAttribute(kfn[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2);
  lc.blockDim = dim3(kGemmThreads);
  lc.dynamicSmemBytes = smem_bytes_of<kGroup>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, (const void*)tc_gemm_kernel<kGroup>, &lc);
  if (e != cudaSuccess) return e;
  *max_pairs = n;
  return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Phase timing (only while profiling is enabled): an event pair per phase.
struct PhaseTimer {
  ttt_mlp* h;
  cudaStream_t st;
  int phase = -1;
  cudaEvent_t a = nullptr;
  void begin(int p) {
    if (!h->profiling) return;
    phase = p;
    cudaEventCreate(&a);
    cudaEventRecord(a, st);
  }
  void end() {
    if (!h->profiling || phase < 0) return;
    cudaEvent_t b;
    cudaEventCreate(&b);
    cudaEventRecord(b, st);
    h->recs.push_back(ttt_mlp::Rec{phase, a, b});
    phase = -1;
  }
};

// `count` consecutive zeroed ints of the control block for one launch
// (count <= kCtrlInts - kCounterBase).
int* next_counters(ttt_mlp* h, cudaStream_t st, int count) {
  if (h->counter_next + count > kCtrlInts) {
    cudaMemsetAsync(h->ctrl + kCounterBase, 0, (kCtrlInts - kCounterBase) * sizeof(int), st);
    h->counter_next = kCounterBase;
  }
  int* p = h->ctrl + h->counter_next;
  h->counter_next += count;
  return p;
}

int* next_counter(ttt_mlp* h, cudaStream_t st) { return next_counters(h, st, 1); }

// Most groups that one group launch chains (TTT_GROUP_RUN overrides, 1..256;
// 1 gives one launch per group).
int group_run() {
  static const int r = [] {
    const char* v = std::getenv("TTT_GROUP_RUN");
    const int n = v ? std::atoi(v) : kMaxGroups;
    return (n >= 1 && n <= kMaxGroups) ? n : kMaxGroups;
  }();
  return r;
}

ttt_status forward_tc(ttt_mlp* h, int doc, const void* x, const void* x0, int64_t n,
                      const std::vector<Span>& groups, void* o, cudaStream_t st) {
  const ttt_mlp_config& c = h->cfg;
  const int d = c.d, f = c.f;
  std::string why;
  CUtensorMap map_x, map_u, map_za, map_zb, map_vmn, map_zmn, map_va;
  if (!make_map(&map_x, x, d, n, d, 64, 128, &why) ||
      !make_map(&map_va, h->V, d, n, d, 64, 128, &why) ||
      !make_map(&map_u, h->U, d, n, d, 64, 128, &why) ||
      !make_map(&map_za, h->Z, f, n, f, 64, 128, &why) ||
      !make_map(&map_zb, h->Z, f, n, f, 64, 128, &why) ||
      !make_map(&map_vmn, h->V, d, n, d, 64, 64, &why) ||
      !make_map(&map_zmn, h->Z, f, n, f, 64, 64, &why))
    return fail(h, TTT_ECUDA, why);

  // fresh tile counters for this call
  TTT_CK(h, cudaMemsetAsync(h->ctrl + kCounterBase, 0, (kCtrlInts - kCounterBase) * sizeof(int), st));
  h->counter_next = kCounterBase;

  PhaseTimer pt{h, st};
  h->prof_calls++;
  // chunk-local Conv1D target source U, wave by wave (<= kMaxSpans groups each)
  pt.begin(0);
  for (size_t w0 = 0; w0 < groups.size(); w0 += kMaxSpans) {
    const size_t w1 = std::min(groups.size(), w0 + kMaxSpans);
    SpanList sl{};
    sl.n = (int)(w1 - w0);
    sl.chunk = c.chunk;
    for (size_t i = w0; i < w1; ++i) {
      sl.start[i - w0] = groups[i].start;
      sl.len[i - w0] = groups[i].len;
    }
    TTT_CK(h, launch_conv(conv_grid<__nv_bfloat16>(sl, d), st, (const __nv_bfloat16*)x0,
                          (const __nv_bfloat16*)h->conv, (__nv_bfloat16*)h->U, d, c.conv_k, sl,
                          c.target_mode));
    h->prof_launches++;
  }
  pt.end();

  GemmArgs a;
  std::memset(&a, 0, sizeof a);
  a.n_rows = (int)n;
  a.d = d;
  a.f = f;
  a.chunk = c.chunk;
  a.err = h->ctrl;
  a.s_pad = h->s_pad;

  // Z = SiLU(X Wg^T) (.) (X Wu^T) for every token of the call (W-independent)
  a.map[0] = map_x;
  a.map[1] = h->map_wg;
  a.map[2] = h->map_wu;
  a.out0 = h->Z;
  a.counter = next_counter(h, st);
  pt.begin(1);
  TTT_CK(h, launch_gemm<kSwiGLU>(h, a, cdiv_h(cdiv_h((int)n, kBM), 2) * cdiv_h(f, kBM), st));
  pt.end();
  h->prof_launches++;

  // V = eta * U W_target for every token
  a.map[0] = map_u;
  a.map[1] = h->map_wtT;
  a.out0 = h->V;
  a.alpha = c.eta;
  a.kdim = d;
  a.counter = next_counter(h, st);
  a.test_withhold_block = fault_injected("kernel_wait") ? 1 : 0;
  pt.begin(2);
  TTT_CK(h, launch_gemm<kLinear>(h, a, cdiv_h(cdiv_h((int)n, kBM), 2) * cdiv_h(d, kBN), st));
  a.test_withhold_block = 0;
  pt.end();
  h->prof_launches++;

  const size_t wsz = (size_t)d * f;
  uint16_t* hi[2] = {h->Whi + (size_t)doc * 2 * wsz, h->Whi + (size_t)doc * 2 * wsz + wsz};
  uint16_t* lo = h->Wlo + (size_t)doc * wsz;
  // the slot's state planes: operand and L2-prefetch boxes (64 x 128), and the
  // update epilogue's boxes (64 x 32) of both planes and of W_0
  CUtensorMap map_hi[2], map_lo, map_hi_e[2], map_lo_e, map_w0_e;
  if (!make_map(&map_hi[0], hi[0], f, d, f, 64, 128, &why) ||
      !make_map(&map_hi[1], hi[1], f, d, f, 64, 128, &why) ||
      !make_map(&map_lo, lo, f, d, f, 64, 128, &why) ||
      !make_map(&map_hi_e[0], hi[0], f, d, f, 64, 32, &why) ||
      !make_map(&map_hi_e[1], hi[1], f, d, f, 64, 32, &why) ||
      !make_map(&map_lo_e, lo, f, d, f, 64, 32, &why) ||
      !make_map(&map_w0_e, h->w0, f, d, f, 64, 32, &why))
    return fail(h, TTT_ECUDA, why);
  for (size_t w0 = 0; w0 < groups.size(); w0 += (size_t)h->s_slots) {
    const size_t w1 = std::min(groups.size(), w0 + (size_t)h->s_slots);
    // intra-group Gram blocks S_g = mask(Z_g Z_g^T) of this wave
    GemmArgs s;
    std::memset(&s, 0, sizeof s);
    s.n_rows = (int)n;
    s.d = d;
    s.f = f;
    s.chunk = c.chunk;
    s.err = h->ctrl;
    s.s_pad = h->s_pad;
    s.n_groups = (int)(w1 - w0);
    for (size_t i = w0; i < w1; ++i) {
      s.g_start[i - w0] = groups[i].start;
      s.g_len[i - w0] = groups[i].len;
    }
    s.map[0] = map_za;
    s.map[1] = map_zb;
    s.out0 = h->S;
    s.counter = next_counter(h, st);
    const int per = cdiv_h(cdiv_h(h->s_pad, kBM), 2) * cdiv_h(h->s_pad, kBN);
    if (c.clip_tau > 0.0f) {
      // per-chunk update clipping: same-chunk Gram blocks of V and Z, then
      // each chunk's rows of V scaled by min(1, tau / ||V_c^T Z_c||_F)
      GemmArgs q = s;
      q.map[0] = map_va;
      q.map[1] = map_va;
      q.f = d;
      q.out0 = h->GV;
      q.counter = next_counter(h, st);
      TTT_CK(h, launch_gemm<kDGram>(h, q, s.n_groups * per, st));
      q.map[0] = map_za;
      q.map[1] = map_za;
      q.f = f;
      q.out0 = h->GZ;
      q.counter = next_counter(h, st);
      TTT_CK(h, launch_gemm<kDGram>(h, q, s.n_groups * per, st));
      GroupList gl{};
      gl.n = s.n_groups;
      gl.chunk = c.chunk;
      gl.G = h->G;
      gl.pitch = h->s_pad;
      for (int i = 0; i < s.n_groups; ++i) {
        gl.start[i] = s.g_start[i];
        gl.len[i] = s.g_len[i];
      }
      clip_scale_kernel<__nv_bfloat16><<<gl.n * gl.G, 256, 0, st>>>(h->GZ, h->GV, (__nv_bfloat16*)h->V, d,
                                                                     c.clip_tau, gl);
      TTT_CK_LAUNCH(h);
      h->prof_launches += 3;
    }
    if (h->G > 1) {
      pt.begin(3);
      TTT_CK(h, launch_gemm<kSGram>(h, s, s.n_groups * per, st));
      pt.end();
      h->prof_launches++;
    }
    pt.begin(4);
    // Runs of consecutive groups, one launch each.  A run ends at a group
    // whose length is not a whole number of K blocks (the update tiles'
    // operand maps are clipped at its end, so the rows past it read zero).
    const int npd = cdiv_h(d, kBN);
    const int run_max = std::min(group_run(), (kCtrlInts - kCounterBase - 1) / (2 * npd));
    if (run_max < 1) return fail(h, TTT_EINVAL, "d too large for the group launch's counters");
    auto exact = [&](size_t k) {
      return groups[k].len % kBK == 0 || (int64_t)groups[k].start + groups[k].len == n;
    };
    for (size_t i = w0; i < w1;) {
      size_t e = i;  // the run's last group
      while (exact(e) && e + 1 < w1 && (int)(e + 1 - i) < run_max) ++e;
      GemmArgs& q = a;
      q.map[0] = map_za;
      q.map[1] = map_hi[0];
      q.map[2] = h->map_s;
      q.map[3] = map_vmn;
      q.map[6] = map_lo;
      q.map[7] = map_hi[1];
      q.map[8] = h->map_w0;
      q.map[9] = map_hi_e[0];
      q.map[10] = map_hi_e[1];
      q.map[11] = map_lo_e;
      q.map[12] = map_w0_e;
      if (exact(e)) {
        q.map[4] = map_vmn;
        q.map[5] = map_zmn;
      } else {
        const uint64_t ext = (uint64_t)groups[e].start + (uint64_t)groups[e].len;
        if (!make_map(&q.map[4], h->V, d, ext, d, 64, 64, &why) ||
            !make_map(&q.map[5], h->Z, f, ext, f, 64, 64, &why))
          return fail(h, TTT_ECUDA, why);
      }
      // per group: its tiles, where its state comes from (W_0 at a document
      // start, else the hi plane the previous group wrote) and where its
      // update tiles write the next hi plane
      q.n_groups = (int)(e - i + 1);
      int cur = h->hcur[doc], tiles = 0;
      for (int k = 0; k < q.n_groups; ++k) {
        const Span& g = groups[i + k];
        q.g_start[k] = g.start;
        q.g_len[k] = g.len;
        q.g_tile[k] = tiles;
        tiles += cdiv_h(cdiv_h(g.len, kBM), 2) * npd + npd * cdiv_h(f, kBN);
        uint8_t fl = 0;
        if (g.reset)
          fl |= kGrpReset;
        else if (cur)
          fl |= kGrpInWb1;
        if (cur ^ 1) fl |= kGrpOutWb1;
        q.g_flags[k] = fl;
        cur ^= 1;
      }
      q.g_tile[q.n_groups] = tiles;
      q.slot0 = (int)(i - w0);
      q.out0 = o;
      int* ctr = next_counters(h, st, 1 + 2 * q.n_groups * npd);
      q.counter = ctr;
      q.dep = ctr + 1;
      // failure-path test hook: the first group launch of the call withholds
      // one of its own operand loads (its bounded waits then run out)
      q.test_withhold_block = (i == 0 && fault_injected("group_wait")) ? 1 : 0;
      TTT_CK(h, launch_gemm<kGroup>(h, q, tiles, st));
      q.test_withhold_block = 0;
      h->prof_launches++;
      h->prof_group_launches++;
      h->hcur[doc] = (uint8_t)cur;
      i = e + 1;
    }
    pt.end();
  }
  return TTT_OK;
}

// The block's static MLP, O = SwiGLU(X) W_0^T, on the tcgen05 path: the
// SwiGLU producer, then O = Z W_0^T with the plain GEMM tiles.  No fast
// weight is read or written.
ttt_status forward_static_tc(ttt_mlp* h, const void* x, int64_t n, void* o, cudaStream_t st) {
  const ttt_mlp_config& c = h->cfg;
  const int d = c.d, f = c.f;
  std::string why;
  CUtensorMap map_x, map_z;
  if (!make_map(&map_x, x, d, n, d, 64, 128, &why) || !make_map(&map_z, h->Z, f, n, f, 64, 128, &why))
    return fail(h, TTT_ECUDA, why);
  TTT_CK(h, cudaMemsetAsync(h->ctrl + kCounterBase, 0, (kCtrlInts - kCounterBase) * sizeof(int), st));
  h->counter_next = kCounterBase;
  GemmArgs a;
  std::memset(&a, 0, sizeof a);
  a.n_rows = (int)n;
  a.d = d;
  a.f = f;
  a.chunk = c.chunk;
  a.err = h->ctrl;
  a.map[0] = map_x;
  a.map[1] = h->map_wg;
  a.map[2] = h->map_wu;
  a.out0 = h->Z;
  a.counter = next_counter(h, st);
  TTT_CK(h, launch_gemm<kSwiGLU>(h, a, cdiv_h(cdiv_h((int)n, kBM), 2) * cdiv_h(f, kBM), st));
  a.map[0] = map_z;
  a.map[1] = h->map_w0;
  a.kdim = f;
  a.alpha = 1.0f;
  a.out0 = o;
  a.counter = next_counter(h, st);
  TTT_CK(h, launch_gemm<kLinear>(h, a, cdiv_h(cdiv_h((int)n, kBM), 2) * cdiv_h(d, kBN), st));
  h->prof_launches += 2;
  return TTT_OK;
}

template <typename T>
ttt_status forward_static_simt(ttt_mlp* h, const void* xv, int64_t n, void* ov, cudaStream_t st) {
  const int d = h->cfg.d, f = h->cfg.f, nn = (int)n;
  float* Z = (float*)h->Z;
  dim3 gz((f + 63) / 64, (nn + 63) / 64);
  simt_swiglu_kernel<T><<<gz, 256, 0, st>>>(nn, f, d, (const T*)xv, (const T*)h->wg, (const T*)h->wu, Z);
  TTT_CK_LAUNCH(h);
  dim3 ga((d + 63) / 64, (nn + 63) / 64);
  simt_gemm_kernel<float, T, T><<<ga, 256, 0, st>>>(nn, d, f, Z, f, 1, (const T*)h->w0, 1, f, (T*)ov, d,
                                                    1.0f, 0.0f);
  TTT_CK_LAUNCH(h);
  h->prof_launches += 2;
  return TTT_OK;
}

template <typename T>
ttt_status forward_simt_t(ttt_mlp* h, int doc, const void* xv, const void* x0v, int64_t n,
                          const std::vector<Span>& spans, void* ov, cudaStream_t st) {
  const ttt_mlp_config& c = h->cfg;
  const int d = c.d, f = c.f;
  const T* x = (const T*)xv;
  const T* x0 = (const T*)x0v;
  T* o = (T*)ov;
  float* Z = (float*)h->Z;
  float* U = (float*)h->U;
  float* V = (float*)h->V;
  const size_t wsz = (size_t)d * f;
  float* W = h->W + (size_t)doc * wsz;
  const int nn = (int)n;

  h->prof_calls++;
  dim3 gz((f + 63) / 64, (nn + 63) / 64);
  simt_swiglu_kernel<T><<<gz, 256, 0, st>>>(nn, f, d, x, (const T*)h->wg, (const T*)h->wu, Z);
  TTT_CK_LAUNCH(h);
  h->prof_launches++;
  for (size_t w0 = 0; w0 < spans.size(); w0 += kMaxSpans) {
    const size_t w1 = std::min(spans.size(), w0 + kMaxSpans);
    SpanList sl{};
    sl.n = (int)(w1 - w0);
    sl.chunk = c.chunk;
    for (size_t i = w0; i < w1; ++i) {
      sl.start[i - w0] = spans[i].start;
      sl.len[i - w0] = spans[i].len;
    }
    TTT_CK(h, launch_conv(conv_grid<T>(sl, d), st, x0, (const T*)h->conv, U, d, c.conv_k, sl, c.target_mode));
    h->prof_launches++;
  }
  dim3 gv((d + 63) / 64, (nn + 63) / 64);
  simt_gemm_kernel<float, T, float><<<gv, 256, 0, st>>>(nn, d, d, U, d, 1, (const T*)h->wt, d, 1, V, d, c.eta, 0.0f);
  TTT_CK_LAUNCH(h);
  h->prof_launches++;
  for (const Span& s : spans) {
    if (s.reset) {
      to_f32_kernel<T><<<grid_for((long long)wsz, 256), 256, 0, st>>>((const T*)h->w0, W, (long long)wsz);
      TTT_CK_LAUNCH(h);
      h->prof_launches++;
    }
    // apply: O_c = Z_c W^T with the state before this chunk's update
    dim3 ga((d + 63) / 64, (s.len + 63) / 64);
    simt_gemm_kernel<float, float, T><<<ga, 256, 0, st>>>(s.len, d, f, Z + (size_t)s.start * f, f, 1, W, 1, f,
                                                          o + (size_t)s.start * d, d, 1.0f, 0.0f);
    TTT_CK_LAUNCH(h);
    if (c.clip_tau > 0.0f) {
      // per-chunk update clipping (Gram form of ||V_c^T Z_c||_F, then V_c scaled)
      dim3 gg((s.len + 63) / 64, (s.len + 63) / 64);
      simt_gemm_kernel<float, float, float><<<gg, 256, 0, st>>>(s.len, s.len, f, Z + (size_t)s.start * f, f, 1,
                                                                Z + (size_t)s.start * f, 1, f, h->GZ, c.chunk,
                                                                1.0f, 0.0f);
      TTT_CK_LAUNCH(h);
      simt_gemm_kernel<float, float, float><<<gg, 256, 0, st>>>(s.len, s.len, d, V + (size_t)s.start * d, d, 1,
                                                                V + (size_t)s.start * d, 1, d, h->GV, c.chunk,
                                                                1.0f, 0.0f);
      TTT_CK_LAUNCH(h);
      GroupList gl{};
      gl.n = 1;
      gl.chunk = c.chunk;
      gl.G = 1;
      gl.pitch = c.chunk;
      gl.start[0] = s.start;
      gl.len[0] = s.len;
      clip_scale_kernel<float><<<1, 256, 0, st>>>(h->GZ, h->GV, V, d, c.clip_tau, gl);
      TTT_CK_LAUNCH(h);
      h->prof_launches += 3;
    }
    // update: W += (eta V_c)^T Z_c
    dim3 gu((f + 63) / 64, (d + 63) / 64);
    simt_gemm_kernel<float, float, float><<<gu, 256, 0, st>>>(d, f, s.len, V + (size_t)s.start * d, 1, d,
                                                              Z + (size_t)s.start * f, f, 1, W, f, 1.0f, 1.0f);
    TTT_CK_LAUNCH(h);
    h->prof_launches += 2;
  }
  return TTT_OK;
}

ttt_status check_handle(const ttt_mlp* h) {
  if (!h) return fail(nullptr, TTT_EINVAL, "handle is NULL");
  return TTT_OK;
}

ttt_status validate_call(ttt_mlp* h, int doc, const void* x, const void* x0, int64_t n,
                         const int64_t* ds, int nds, const void* o) {
  const ttt_mlp_config& c = h->cfg;
  if (doc < 0 || doc >= c.n_docs) return fail(h, TTT_EINVAL, "doc slot out of range");
  if (n < 0 || n > c.max_tokens) return fail(h, TTT_EINVAL, "n_tokens must be in 0..max_tokens");
  if (nds < 0 || (nds > 0 && !ds)) return fail(h, TTT_EINVAL, "doc_starts is NULL but n_doc_starts > 0");
  for (int i = 0; i < nds; ++i) {
    if (ds[i] < 0 || ds[i] >= std::max<int64_t>(n, 1) || (n == 0))
      return fail(h, TTT_EINVAL, "document starts must lie in [0, n_tokens)");
    if (i > 0 && ds[i] <= ds[i - 1]) return fail(h, TTT_EINVAL, "document starts must be strictly increasing");
  }
  if (n == 0) return TTT_OK;
  if (!x || !x0 || !o) return fail(h, TTT_EINVAL, "x, x0 and o must be non-NULL");
  if (!aligned16(x) || !aligned16(x0) || !aligned16(o)) return fail(h, TTT_EINVAL, "x, x0 and o must be 16-byte aligned");
  const size_t bytes = (size_t)n * c.d * (c.act_dtype == TTT_BF16 ? 2 : 4);
  auto overlap = [&](const void* p, const void* q) {
    const uintptr_t a0 = (uintptr_t)p, b0 = (uintptr_t)q;
    return a0 < b0 + bytes && b0 < a0 + bytes;
  };
  if (overlap(o, x) || overlap(o, x0)) return fail(h, TTT_EINVAL, "o must not overlap x or x0");
  return TTT_OK;
}

ttt_status forward_impl(ttt_mlp* h, int doc, const void* x, const void* x0, int64_t n,
                        const int64_t* ds, int nds, void* o, cudaStream_t st) {
  if (n == 0) return TTT_OK;
  if (h->tc) {
    std::vector<Span> groups = plan_groups(n, h->cfg.chunk, h->G, ds, nds);
    return forward_tc(h, doc, x, x0, n, groups, o, st);
  }
  std::vector<Span> spans = plan_groups(n, h->cfg.chunk, 1, ds, nds);
  if (h->cfg.act_dtype == TTT_BF16)
    return forward_simt_t<__nv_bfloat16>(h, doc, x, x0, n, spans, o, st);
  return forward_simt_t<float>(h, doc, x, x0, n, spans, o, st);
}

// Tokens per segment of a host-buffer call (TTT_HOST_SEGMENT overrides it,
// at least 256).
int64_t host_segment_tokens() {
  static const int64_t n = [] {
    const char* v = std::getenv("TTT_HOST_SEGMENT");
    const long long t = v ? std::atoll(v) : 8192;
    return (int64_t)(t >= 256 ? t : 8192);
  }();
  return n;
}

// Where a host-buffer call is cut into segments: at group starts (chunk
// starts on the fp32 path), every segment at least host_segment_tokens() long
// except the last, which is the call's last group alone (its output copy is
// the one no layer overlaps, so it is kept short).  On a handle with a shared
// scratch the first segment is half as long as the others (its input copy
// cannot overlap the previous call there).  A segment that starts at a group
// start and runs as a call of its own makes the same chunks and groups, and so
// the same bits, as the whole call: a group start is a chunk start, the conv
// window never crosses a chunk, and the slot's state carries over.
std::vector<int64_t> host_cuts(ttt_mlp* h, int64_t n, const int64_t* ds, int nds) {
  const std::vector<Span> groups = plan_groups(n, h->cfg.chunk, h->tc ? h->G : 1, ds, nds);
  const int64_t seg = host_segment_tokens();
  const int64_t first = h->owns_scratch ? seg : seg / 2;
  std::vector<int64_t> cuts{0};
  for (const Span& g : groups)
    if (g.start - cuts.back() >= (cuts.size() == 1 ? first : seg)) cuts.push_back(g.start);
  if (groups.size() > 1 && groups.back().start > cuts.back()) cuts.push_back(groups.back().start);
  cuts.push_back(n);
  return cuts;
}

ttt_status reset_slot(ttt_mlp* h, int doc, cudaStream_t st) {
  const size_t wsz = (size_t)h->cfg.d * h->cfg.f;
  if (h->tc) {
    // W_0 is bf16: its hi plane is W_0's bits and its lo plane is zero
    TTT_CK(h, cudaMemcpyAsync(h->Whi + (size_t)doc * 2 * wsz + h->hcur[doc] * wsz, h->w0, wsz * 2,
                              cudaMemcpyDeviceToDevice, st));
    TTT_CK(h, cudaMemsetAsync(h->Wlo + (size_t)doc * wsz, 0, wsz * 2, st));
    return TTT_OK;
  }
  float* W = h->W + (size_t)doc * wsz;
  if (h->cfg.act_dtype == TTT_BF16)
    to_f32_kernel<__nv_bfloat16><<<grid_for((long long)wsz, 256), 256, 0, st>>>((const __nv_bfloat16*)h->w0, W, (long long)wsz);
  else
    to_f32_kernel<float><<<grid_for((long long)wsz, 256), 256, 0, st>>>((const float*)h->w0, W, (long long)wsz);
  TTT_CK_LAUNCH(h);
  return TTT_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

size_t ttt_mlp_workspace_bytes(const ttt_mlp_config* cfg) {
  std::string why;
  if (!config_ok(cfg, &why)) return 0;
  return align_up(state_bytes_of(*cfg), 256) + scratch_bytes_of(*cfg);
}

size_t ttt_mlp_state_bytes(const ttt_mlp_config* cfg) {
  std::string why;
  if (!config_ok(cfg, &why)) return 0;
  return state_bytes_of(*cfg);
}

size_t ttt_mlp_scratch_bytes(const ttt_mlp_config* cfg) {
  std::string why;
  if (!config_ok(cfg, &why)) return 0;
  return scratch_bytes_of(*cfg);
}

ttt_status ttt_mlp_create_split(const ttt_mlp_config* cfg, const void* w_gate, const void* w_up,
                                const void* w_down0, const void* conv_w, const void* w_target,
                                void* state, size_t state_bytes, void* scratch, size_t scratch_bytes,
                                void* stream, ttt_mlp** out) {
  if (fault_injected("create")) return fail(nullptr, TTT_EFAULT_INJECTED, "fault injected: create");
  if (!out) return fail(nullptr, TTT_EINVAL, "out is NULL");
  *out = nullptr;
  std::string why;
  if (!config_ok(cfg, &why)) return fail(nullptr, TTT_EINVAL, why);
  const void* ptrs[5] = {w_gate, w_up, w_down0, conv_w, w_target};
  for (const void* p : ptrs) {
    if (!p) return fail(nullptr, TTT_EINVAL, "weight pointers must be non-NULL");
    if (!aligned16(p)) return fail(nullptr, TTT_EINVAL, "weight pointers must be 16-byte aligned");
  }
  if (!state || (reinterpret_cast<uintptr_t>(state) & 255u) || !scratch ||
      (reinterpret_cast<uintptr_t>(scratch) & 255u))
    return fail(nullptr, TTT_EINVAL, "state and scratch must be non-NULL and 256-byte aligned");
  const bool tc = tc_shape_ok(*cfg) && !force_simt();
  const Layout l = make_layout(*cfg, tc);
  if (state_bytes < l.state_total || scratch_bytes < l.scratch_total)
    return fail(nullptr, TTT_EINVAL, "state or scratch is smaller than ttt_mlp_state_bytes() / ttt_mlp_scratch_bytes()");
  {
    const uintptr_t a0 = (uintptr_t)state, b0 = (uintptr_t)scratch;
    if (a0 < b0 + l.scratch_total && b0 < a0 + l.state_total)
      return fail(nullptr, TTT_EINVAL, "state and scratch must not overlap");
  }

  ttt_mlp* h = new ttt_mlp();
  h->cfg = *cfg;
  h->wg = w_gate;
  h->wu = w_up;
  h->w0 = w_down0;
  h->conv = conv_w;
  h->wt = w_target;
  h->tc = tc;
  h->G = l.G;
  h->L = l.L;
  h->s_pad = l.s_pad;
  h->s_slots = l.s_slots;
  uint8_t* sb = (uint8_t*)state;
  uint8_t* xb = (uint8_t*)scratch;
  h->ctrl = (int*)(sb + l.ctrl);
  h->W = tc ? nullptr : (float*)(sb + l.W);
  h->Whi = tc ? (uint16_t*)(sb + l.Whi) : nullptr;
  h->Wlo = tc ? (uint16_t*)(sb + l.Wlo) : nullptr;
  h->hcur.assign((size_t)cfg->n_docs, 0);
  h->WtT = (__nv_bfloat16*)(sb + l.WtT);
  h->Z = xb + l.Z;
  h->U = xb + l.U;
  h->V = xb + l.V;
  h->S = (__nv_bfloat16*)(xb + l.S);
  h->GZ = l.GZ ? (float*)(xb + l.GZ) : nullptr;
  h->GV = l.GV ? (float*)(xb + l.GV) : nullptr;
  h->xs = xb + l.xs;
  h->x0s = xb + l.x0s;
  h->os = xb + l.os;
  h->xs2 = xb + l.xs2;
  h->x0s2 = xb + l.x0s2;
  h->counter_next = kCounterBase;
  cudaStream_t st = (cudaStream_t)stream;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    std::string m = std::string("cudaGetDevice/attribute: ") + cudaGetErrorString(e);
    delete h;
    return fail(nullptr, TTT_ECUDA, m);
  }
  auto bail = [&](ttt_status s, const std::string& m) {
    delete h;
    return fail(nullptr, s, m);
  };
  if (tc) {
    const int d = cfg->d, f = cfg->f;
    if (!make_map(&h->map_wg, w_gate, d, f, d, 64, 128, &why) ||
        !make_map(&h->map_wu, w_up, d, f, d, 64, 128, &why) ||
        !make_map(&h->map_wtT, h->WtT, d, d, d, 64, 128, &why) ||
        !make_map(&h->map_s, h->S, h->s_pad, (uint64_t)h->s_slots * h->s_pad, h->s_pad, 64, 128, &why) ||
        !make_map(&h->map_w0, w_down0, f, d, f, 64, 128, &why))
      return bail(TTT_ECUDA, why);
    e = setup_tc_kernels(&h->max_pairs);
    if (e != cudaSuccess)
      return bail(TTT_ECUDA, std::string("tcgen05 kernel set-up (attributes, cluster occupancy): ") +
                                 cudaGetErrorString(e));
    dim3 tb(32, 8), tg((d + 31) / 32, (d + 31) / 32);
    transpose_kernel<__nv_bfloat16><<<tg, tb, 0, st>>>((const __nv_bfloat16*)w_target, h->WtT, d, d);
    e = cudaGetLastError();
    if (e != cudaSuccess) return bail(TTT_ECUDA, std::string("transpose launch: ") + cudaGetErrorString(e));
  }
  e = cudaMemsetAsync(h->ctrl, 0, kCtrlInts * sizeof(int), st);
  if (e != cudaSuccess) return bail(TTT_ECUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  for (int s = 0; s < cfg->n_docs; ++s) {
    if (reset_slot(h, s, st) != TTT_OK) {
      std::string m = h->err;
      delete h;
      return fail(nullptr, TTT_ECUDA, m);
    }
  }
  *out = h;
  return TTT_OK;
}

ttt_status ttt_mlp_create(const ttt_mlp_config* cfg, const void* w_gate, const void* w_up,
                          const void* w_down0, const void* conv_w, const void* w_target,
                          void* workspace, size_t workspace_bytes, void* stream, ttt_mlp** out) {
  if (fault_injected("create")) return fail(nullptr, TTT_EFAULT_INJECTED, "fault injected: create");
  if (!out) return fail(nullptr, TTT_EINVAL, "out is NULL");
  *out = nullptr;
  std::string why;
  if (!config_ok(cfg, &why)) return fail(nullptr, TTT_EINVAL, why);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(nullptr, TTT_EINVAL, "workspace must be non-NULL and 256-byte aligned");
  // the workspace is the state part followed by the scratch part
  const size_t sb = align_up(state_bytes_of(*cfg), 256), xb = scratch_bytes_of(*cfg);
  if (workspace_bytes < sb + xb) return fail(nullptr, TTT_EINVAL, "workspace is smaller than ttt_mlp_workspace_bytes()");
  ttt_status r = ttt_mlp_create_split(cfg, w_gate, w_up, w_down0, conv_w, w_target, workspace, sb,
                                      (uint8_t*)workspace + sb, workspace_bytes - sb, stream, out);
  if (r == TTT_OK) (*out)->owns_scratch = true;
  return r;
}

ttt_status ttt_mlp_forward_chunks(ttt_mlp* h, int32_t doc, const void* x, const void* x0,
                                  int64_t n_tokens, const int64_t* doc_starts,
                                  int32_t n_doc_starts, void* o, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("forward")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: forward");
  ttt_status s = validate_call(h, doc, x, x0, n_tokens, doc_starts, n_doc_starts, o);
  if (s != TTT_OK) return s;
  return forward_impl(h, doc, x, x0, n_tokens, doc_starts, n_doc_starts, o, (cudaStream_t)stream);
}

ttt_status ttt_mlp_forward_static(ttt_mlp* h, const void* x, int64_t n_tokens, void* o, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("forward")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: forward");
  ttt_status s = validate_call(h, 0, x, x, n_tokens, nullptr, 0, o);
  if (s != TTT_OK || n_tokens == 0) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->tc) return forward_static_tc(h, x, n_tokens, o, st);
  if (h->cfg.act_dtype == TTT_BF16) return forward_static_simt<__nv_bfloat16>(h, x, n_tokens, o, st);
  return forward_static_simt<float>(h, x, n_tokens, o, st);
}

ttt_status ttt_mlp_forward_chunks_host(ttt_mlp* h, int32_t doc, const void* x_host,
                                       const void* x0_host, int64_t n_tokens,
                                       const int64_t* doc_starts, int32_t n_doc_starts,
                                       void* o_host, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("forward")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: forward");
  if (n_tokens > 0 && (!x_host || !x0_host || !o_host))
    return fail(h, TTT_EINVAL, "host buffers must be non-NULL");
  ttt_status s = validate_call(h, doc, h->xs, h->x0s, n_tokens, doc_starts, n_doc_starts, h->os);
  if (s != TTT_OK || n_tokens == 0) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (!h->st_in) {
    TTT_CK(h, cudaStreamCreateWithFlags(&h->st_in, cudaStreamNonBlocking));
    TTT_CK(h, cudaStreamCreateWithFlags(&h->st_out, cudaStreamNonBlocking));
    for (cudaEvent_t* e : {&h->ev_start, &h->ev_in, &h->ev_out, &h->ev_free[0], &h->ev_free[1]})
      TTT_CK(h, cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  }
  // Segments pipelined over three streams: segment k+1's input copy (st_in)
  // and segment k-1's output copy (st_out) overlap segment k's layer on
  // `stream`.  Events order them, and `stream` finally waits for the last
  // output copy.  The output copies first wait for everything already on
  // `stream`.  The input copies wait only until the staging buffers they
  // fill are free: with a scratch of its own the handle alternates two pairs
  // of them between calls, so a call's input copies need only the layers of
  // the call before the previous one to be done and overlap the previous
  // call; with a shared scratch they wait for everything already on `stream`.
  const size_t tok = (size_t)h->cfg.d * (h->cfg.act_dtype == TTT_BF16 ? 2 : 4);
  const bool sep_x0 = x0_host != x_host;
  const int buf = h->owns_scratch ? h->stage_sel : 0;
  void* xs = buf ? h->xs2 : h->xs;
  void* x0s = buf ? h->x0s2 : h->x0s;
  const std::vector<int64_t> cuts = host_cuts(h, n_tokens, doc_starts, n_doc_starts);
  auto copy_in = [&](size_t k) -> ttt_status {
    const size_t off = (size_t)cuts[k] * tok, len = (size_t)(cuts[k + 1] - cuts[k]) * tok;
    TTT_CK(h, cudaMemcpyAsync((char*)xs + off, (const char*)x_host + off, len, cudaMemcpyHostToDevice, h->st_in));
    if (sep_x0)
      TTT_CK(h, cudaMemcpyAsync((char*)x0s + off, (const char*)x0_host + off, len, cudaMemcpyHostToDevice,
                                h->st_in));
    TTT_CK(h, cudaEventRecord(h->ev_in, h->st_in));
    return TTT_OK;
  };
  TTT_CK(h, cudaEventRecord(h->ev_start, st));
  TTT_CK(h, cudaStreamWaitEvent(h->st_in, h->owns_scratch ? h->ev_free[buf] : h->ev_start, 0));
  TTT_CK(h, cudaStreamWaitEvent(h->st_out, h->ev_start, 0));
  // On any return from here on, mark the staging buffers as read by what
  // this call has enqueued on `stream`, so that a later call never fills them
  // under layers still in flight.
  struct MarkFree {
    ttt_mlp* h;
    int buf;
    cudaStream_t st;
    bool armed = true;
    ~MarkFree() {
      if (armed) cudaEventRecord(h->ev_free[buf], st);
    }
  } mark{h, buf, st};
  if ((s = copy_in(0)) != TTT_OK) return s;
  for (size_t k = 0; k + 1 < cuts.size(); ++k) {
    const int64_t b = cuts[k], e = cuts[k + 1];
    TTT_CK(h, cudaStreamWaitEvent(st, h->ev_in, 0));  // input k has landed
    if (k + 2 < cuts.size() && (s = copy_in(k + 1)) != TTT_OK) return s;
    std::vector<int64_t> dsk;
    for (int i = 0; i < n_doc_starts; ++i)
      if (doc_starts[i] >= b && doc_starts[i] < e) dsk.push_back(doc_starts[i] - b);
    const size_t off = (size_t)b * tok;
    s = forward_impl(h, doc, (char*)xs + off, (char*)(sep_x0 ? x0s : xs) + off, e - b, dsk.data(),
                     (int)dsk.size(), (char*)h->os + off, st);
    if (s != TTT_OK) return s;
    TTT_CK(h, cudaEventRecord(h->ev_out, st));
    TTT_CK(h, cudaStreamWaitEvent(h->st_out, h->ev_out, 0));
    TTT_CK(h, cudaMemcpyAsync((char*)o_host + off, (char*)h->os + off, (size_t)(e - b) * tok,
                              cudaMemcpyDeviceToHost, h->st_out));
  }
  // the layers that read this call's staging buffers are enqueued
  mark.armed = false;
  TTT_CK(h, cudaEventRecord(h->ev_free[buf], st));
  if (h->owns_scratch) h->stage_sel ^= 1;
  TTT_CK(h, cudaEventRecord(h->ev_out, h->st_out));
  TTT_CK(h, cudaStreamWaitEvent(st, h->ev_out, 0));
  return TTT_OK;
}

ttt_status ttt_mlp_reset(ttt_mlp* h, int32_t doc, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("reset")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: reset");
  if (doc < -1 || doc >= h->cfg.n_docs) return fail(h, TTT_EINVAL, "doc slot out of range");
  for (int s = (doc < 0 ? 0 : doc); s < (doc < 0 ? h->cfg.n_docs : doc + 1); ++s) {
    ttt_status r = reset_slot(h, s, (cudaStream_t)stream);
    if (r != TTT_OK) return r;
  }
  return TTT_OK;
}

ttt_status ttt_mlp_get_fast_weight(ttt_mlp* h, int32_t doc, float* dst, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("get")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: get");
  if (doc < 0 || doc >= h->cfg.n_docs) return fail(h, TTT_EINVAL, "doc slot out of range");
  if (!dst) return fail(h, TTT_EINVAL, "dst is NULL");
  const size_t wsz = (size_t)h->cfg.d * h->cfg.f;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->tc) {
    join_planes_kernel<<<grid_for((long long)wsz, 256), 256, 0, st>>>(
        h->Whi + (size_t)doc * 2 * wsz + h->hcur[doc] * wsz, h->Wlo + (size_t)doc * wsz, dst, (long long)wsz);
    TTT_CK_LAUNCH(h);
    return TTT_OK;
  }
  TTT_CK(h, cudaMemcpyAsync(dst, h->W + (size_t)doc * wsz, wsz * 4, cudaMemcpyDeviceToDevice, st));
  return TTT_OK;
}

ttt_status ttt_mlp_set_fast_weight(ttt_mlp* h, int32_t doc, const float* src, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("set")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: set");
  if (doc < 0 || doc >= h->cfg.n_docs) return fail(h, TTT_EINVAL, "doc slot out of range");
  if (!src) return fail(h, TTT_EINVAL, "src is NULL");
  const size_t wsz = (size_t)h->cfg.d * h->cfg.f;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->tc) {
    split_planes_kernel<<<grid_for((long long)wsz, 256), 256, 0, st>>>(
        src, h->Whi + (size_t)doc * 2 * wsz + h->hcur[doc] * wsz, h->Wlo + (size_t)doc * wsz, (long long)wsz);
    TTT_CK_LAUNCH(h);
    return TTT_OK;
  }
  TTT_CK(h, cudaMemcpyAsync(h->W + (size_t)doc * wsz, src, wsz * 4, cudaMemcpyDeviceToDevice, st));
  return TTT_OK;
}

ttt_status ttt_mlp_check(ttt_mlp* h, void* stream) {
  if (check_handle(h)) return TTT_EINVAL;
  if (fault_injected("check")) return fail(h, TTT_EFAULT_INJECTED, "fault injected: check");
  cudaStream_t st = (cudaStream_t)stream;
  TTT_CK(h, cudaStreamSynchronize(st));
  int word = 0;
  TTT_CK(h, cudaMemcpy(&word, h->ctrl, sizeof(int), cudaMemcpyDeviceToHost));
  if (word != 0) {
    TTT_CK(h, cudaMemset(h->ctrl, 0, sizeof(int)));
    static const char* const kWaitNames[] = {"?", "operand stage full", "operand stage empty",
                                             "accumulator full", "accumulator empty",
                                             "tile scheduler", "drain", "completion counter"};
    char buf[128];
    std::snprintf(buf, sizeof buf, "an in-kernel wait ran out (code %d: %s)", word,
                  kWaitNames[(word >= 1 && word <= 7) ? word : 0]);
    return fail(h, TTT_ETIMEOUT, buf);
  }
  return TTT_OK;
}

ttt_status ttt_mlp_destroy(ttt_mlp* h) {
  if (!h) return fail(nullptr, TTT_EINVAL, "handle is NULL");
  ttt_mlp_profile_enable(h, 0);
  delete h;
  return TTT_OK;
}

const char* ttt_mlp_last_error(const ttt_mlp* h) { return h ? h->err.c_str() : g_err.c_str(); }

ttt_status ttt_mlp_intermediates(const ttt_mlp* h, const void** z, const void** v, int32_t* dtype) {
  if (!h || !z || !v || !dtype) return fail(nullptr, TTT_EINVAL, "ttt_mlp_intermediates: NULL argument");
  *z = h->Z;
  *v = h->V;
  *dtype = h->tc ? TTT_BF16 : TTT_F32;
  return TTT_OK;
}

ttt_status ttt_mlp_profile_enable(ttt_mlp* h, int32_t enable) {
  if (check_handle(h)) return TTT_EINVAL;
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  h->recs.clear();
  h->prof_calls = h->prof_group_launches = h->prof_launches = 0;
  h->profiling = enable != 0;
  return TTT_OK;
}

ttt_status ttt_mlp_profile_read(ttt_mlp* h, float* ms, int64_t* counts) {
  if (check_handle(h)) return TTT_EINVAL;
  if (!ms || !counts) return fail(h, TTT_EINVAL, "ttt_mlp_profile_read: NULL argument");
  for (int i = 0; i < 5; ++i) ms[i] = 0.0f;
  for (auto& r : h->recs) {
    TTT_CK(h, cudaEventSynchronize(r.b));
    float t = 0.0f;
    TTT_CK(h, cudaEventElapsedTime(&t, r.a, r.b));
    if (r.phase >= 0 && r.phase < 5) ms[r.phase] += t;
  }
  counts[0] = h->prof_calls;
  counts[1] = h->prof_group_launches;
  counts[2] = h->prof_launches;
  return TTT_OK;
}

const char* ttt_mlp_path(const ttt_mlp* h) { return (h && h->tc) ? "tcgen05" : "simt"; }

ttt_status ttt_rmsnorm(const float* hs, void* x, int64_t n, int32_t d, float eps, int32_t out_dtype,
                       void* stream) {
  if (n < 0 || d < 1 || (n > 0 && (!hs || !x)) || (out_dtype != TTT_F32 && out_dtype != TTT_BF16))
    return fail(nullptr, TTT_EINVAL, "ttt_rmsnorm: bad arguments");
  if (n == 0) return TTT_OK;
  if (n > (int64_t(1) << 31) - 1) return fail(nullptr, TTT_EUNSUPPORTED, "ttt_rmsnorm: too many rows");
  cudaStream_t st = (cudaStream_t)stream;
  if (out_dtype == TTT_BF16)
    rmsnorm_kernel<__nv_bfloat16><<<(unsigned)n, 256, 0, st>>>(hs, (__nv_bfloat16*)x, d, eps);
  else
    rmsnorm_kernel<float><<<(unsigned)n, 256, 0, st>>>(hs, (float*)x, d, eps);
  TTT_CK(nullptr, cudaGetLastError());
  return TTT_OK;
}

ttt_status ttt_residual_add(float* hs, const void* o, int64_t n, int32_t d, int32_t o_dtype, void* stream) {
  if (n < 0 || d < 1 || (n > 0 && (!hs || !o)) || (o_dtype != TTT_F32 && o_dtype != TTT_BF16))
    return fail(nullptr, TTT_EINVAL, "ttt_residual_add: bad arguments");
  if (n == 0) return TTT_OK;
  const long long cnt = n * (long long)d;
  cudaStream_t st = (cudaStream_t)stream;
  if (o_dtype == TTT_BF16)
    residual_add_kernel<__nv_bfloat16><<<grid_for(cnt, 256), 256, 0, st>>>(hs, (const __nv_bfloat16*)o, cnt);
  else
    residual_add_kernel<float><<<grid_for(cnt, 256), 256, 0, st>>>(hs, (const float*)o, cnt);
  TTT_CK(nullptr, cudaGetLastError());
  return TTT_OK;
}

ttt_status ttt_residual_rmsnorm(float* hs, const void* o, void* x, int64_t n, int32_t d, float eps,
                                int32_t o_dtype, int32_t x_dtype, void* stream) {
  if (n < 0 || d < 1 || (n > 0 && (!hs || !o || !x)) || (o_dtype != TTT_F32 && o_dtype != TTT_BF16) ||
      (x_dtype != TTT_F32 && x_dtype != TTT_BF16))
    return fail(nullptr, TTT_EINVAL, "ttt_residual_rmsnorm: bad arguments");
  if (n == 0) return TTT_OK;
  if (n > (int64_t(1) << 31) - 1) return fail(nullptr, TTT_EUNSUPPORTED, "ttt_residual_rmsnorm: too many rows");
  cudaStream_t st = (cudaStream_t)stream;
  const unsigned rows = (unsigned)n;
  if (o_dtype == TTT_BF16 && x_dtype == TTT_BF16)
    residual_rmsnorm_kernel<__nv_bfloat16, __nv_bfloat16><<<rows, 256, 0, st>>>(
        hs, (const __nv_bfloat16*)o, (__nv_bfloat16*)x, d, eps);
  else if (o_dtype == TTT_BF16)
    residual_rmsnorm_kernel<__nv_bfloat16, float><<<rows, 256, 0, st>>>(hs, (const __nv_bfloat16*)o, (float*)x, d, eps);
  else if (x_dtype == TTT_BF16)
    residual_rmsnorm_kernel<float, __nv_bfloat16><<<rows, 256, 0, st>>>(hs, (const float*)o, (__nv_bfloat16*)x, d, eps);
  else
    residual_rmsnorm_kernel<float, float><<<rows, 256, 0, st>>>(hs, (const float*)o, (float*)x, d, eps);
  TTT_CK(nullptr, cudaGetLastError());
  return TTT_OK;
}

}  // extern "C"

// ====================================================================== allocation-free target

// Scratch of ttt_target_noalloc: one file-scope device array per GPU that
// loads the library.  Host code only ever sees a host-side stand-in for this
// name, so the device address is looked up once per device and passed in.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TTT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kNoallocMaxDevices] = {};
int g_noalloc_pairs[kNoallocMaxDevices] = {};

// One-time set-up of the current device: scratch address, kernel attributes
// and the number of co-resident CTA pairs.
ttt_status noalloc_setup(int dev, unsigned char** ptr, int* pairs_out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return fail(nullptr, TTT_ECUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    int pairs = 0;
    e = setup_tc_kernels(&pairs);
    if (e != cudaSuccess)
      return fail(nullptr, TTT_ECUDA, std::string("tcgen05 kernel set-up: ") + cudaGetErrorString(e));
    g_noalloc_pairs[dev] = pairs;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *ptr = g_noalloc_ptr[dev];
  *pairs_out = g_noalloc_pairs[dev];
  return TTT_OK;
}

}  // namespace

extern "C" ttt_status ttt_target_noalloc(const void* x0, const void* conv_w, const void* w_target,
                                         int64_t n_tokens, int32_t d, int32_t conv_k, int32_t chunk,
                                         const int64_t* doc_starts, int32_t n_doc_starts, float eta,
                                         void* v, int32_t* status, void* stream) {
  if (d < 256 || d % 64) return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: d must be a multiple of 64, >= 256");
  if (chunk < 1 || chunk > 1024) return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: chunk must be in 1..1024");
  if (conv_k < 1 || conv_k > 8) return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: conv_k must be in 1..8");
  if (n_tokens < 0 || !std::isfinite(eta)) return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: bad n_tokens or eta");
  if (n_doc_starts < 0 || (n_doc_starts > 0 && !doc_starts))
    return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: doc_starts is NULL but n_doc_starts > 0");
  for (int i = 0; i < n_doc_starts; ++i) {
    if (doc_starts[i] < 0 || doc_starts[i] >= n_tokens || (i > 0 && doc_starts[i] <= doc_starts[i - 1]))
      return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: document starts must be strictly increasing in [0, n_tokens)");
  }
  const uint64_t need = 2ull * d * d + 2ull * (uint64_t)n_tokens * d + 512;
  if (need > TTT_NOALLOC_SCRATCH_BYTES) {
    char buf[200];
    std::snprintf(buf, sizeof buf,
                  "ttt_target_noalloc: needs %llu scratch bytes (2*d*d + 2*n_tokens*d + 512), more than the "
                  "fixed %u-byte array", (unsigned long long)need, (unsigned)TTT_NOALLOC_SCRATCH_BYTES);
    return fail(nullptr, TTT_EUNSUPPORTED, buf);
  }
  if (n_tokens == 0) return TTT_OK;
  if (!x0 || !conv_w || !w_target || !v) return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: NULL buffer");
  if (!aligned16(x0) || !aligned16(conv_w) || !aligned16(w_target) || !aligned16(v))
    return fail(nullptr, TTT_EINVAL, "ttt_target_noalloc: buffers must be 16-byte aligned");

  int dev = 0;
  TTT_CK(nullptr, cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoallocMaxDevices) return fail(nullptr, TTT_EUNSUPPORTED, "ttt_target_noalloc: device ordinal too large");
  unsigned char* scratch = nullptr;
  int pairs = 0;
  ttt_status s = noalloc_setup(dev, &scratch, &pairs);
  if (s != TTT_OK) return s;

  // scratch layout: [0,256) control (tile counter, error word) | W_target^T | U
  int* ctrl = reinterpret_cast<int*>(scratch);
  __nv_bfloat16* wtT = reinterpret_cast<__nv_bfloat16*>(scratch + 256);
  __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(scratch + 256 + align_up(2ull * d * d, 256));
  int* err = status ? status : ctrl + 1;
  cudaStream_t st = (cudaStream_t)stream;

  TTT_CK(nullptr, cudaMemsetAsync(ctrl, 0, 256, st));
  if (status) TTT_CK(nullptr, cudaMemsetAsync(status, 0, sizeof(int32_t), st));
  dim3 tb(32, 8), tg((d + 31) / 32, (d + 31) / 32);
  transpose_kernel<__nv_bfloat16><<<tg, tb, 0, st>>>((const __nv_bfloat16*)w_target, wtT, d, d);
  TTT_CK(nullptr, cudaGetLastError());

  std::vector<Span> docs = plan_groups(n_tokens, chunk, 1 << 30, doc_starts, n_doc_starts);
  for (size_t w0 = 0; w0 < docs.size(); w0 += kMaxSpans) {
    const size_t w1 = std::min(docs.size(), w0 + kMaxSpans);
    SpanList sl{};
    sl.n = (int)(w1 - w0);
    sl.chunk = chunk;
    for (size_t i = w0; i < w1; ++i) {
      sl.start[i - w0] = docs[i].start;
      sl.len[i - w0] = docs[i].len;
    }
    TTT_CK(nullptr, launch_conv(conv_grid<__nv_bfloat16>(sl, d), st, (const __nv_bfloat16*)x0,
                                (const __nv_bfloat16*)conv_w, u, d, conv_k, sl, /*mode=*/0));
  }

  std::string why;
  GemmArgs a;
  std::memset(&a, 0, sizeof a);
  if (!make_map(&a.map[0], u, d, n_tokens, d, 64, 128, &why) ||
      !make_map(&a.map[1], wtT, d, d, d, 64, 128, &why))
    return fail(nullptr, TTT_ECUDA, why);
  a.n_rows = (int)n_tokens;
  a.d = d;
  a.f = d;
  a.kdim = d;
  a.chunk = chunk;
  a.alpha = eta;
  a.counter = ctrl;
  a.err = err;
  a.out0 = v;
  const int npairs = cdiv_h(cdiv_h((int)n_tokens, kBM), 2) * cdiv_h(d, kBN);
  TTT_CK(nullptr, launch_pairs<kLinear>(pairs, a, npairs, st));
  return TTT_OK;
}
