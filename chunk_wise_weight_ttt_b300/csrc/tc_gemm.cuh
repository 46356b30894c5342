// Persistent, warp-specialised tcgen05 GEMM engine for the bf16 hot path.
//
// CTAs run in clusters of two (one CTA per SM) that compute one 256x256 tile
// with the pair form of the 5th-generation MMA (tcgen05 cta_group::2): CTA r
// holds rows [128r, 128r+128) of the A block and of the B block (B's N half)
// in its shared memory, the even CTA issues the MMAs for both, and each CTA's
// TMEM receives its 128 accumulator rows.  A ring stage is therefore 32 KB per
// CTA and carries 1.5x the MMA work per byte of a 128x256 tile.  The group
// kernel has 5 stages plus two state-slice buffers per epilogue warp for its
// update tiles (a sixth stage measured no faster); the other modes have 7.
// The even CTA (the leader) claims tiles from a dynamic counter and hands each
// to its peer through distributed shared memory; both CTAs' TMA loads signal
// the leader's ring barriers, and the leader's commits release the stages and
// accumulators in both CTAs.
//
// Each CTA has 192 threads:
//   warp 0      TMA producer: streams this CTA's operand halves (64 K-elements
//               per block) into its shared-memory ring with 128-byte swizzle.
//   warp 1      owns the TMEM allocation (512 columns = two 128x256 fp32
//               accumulators, allocated together with the peer) and, in the
//               leader, issues the pair's tcgen05.mma from one thread.
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (one TMEM
//               lane = one output row per thread), the mode's arithmetic, and
//               the stores (through TMA for the group kernel's fast-weight
//               state, plain global stores otherwise); the other accumulator
//               is filled meanwhile.
//
// Modes (what the tiles are):
//   kSwiGLU  Z = SiLU(X Wg^T) (.) (X Wu^T): the B tile stacks 128 rows of Wg
//            and the same 128 rows of Wu, so one 128x256 accumulator holds the
//            gate and up halves of a 128x128 block of Z.
//   kLinear  out = alpha * (A B^T) over a K range of `kdim`: the target
//            projection V = eta * (U W_target) (A = U, the chunk-local Conv1D
//            output, B = W_target^T, K = d) and the static MLP's down
//            projection O = Z W_0^T (A = Z, B = W_0, K = f).
//   kSGram   per group of chunks, S = Z_g Z_g^T with every entry whose column
//            chunk is not strictly before its row chunk set to zero.
//   kDGram   per group of chunks, the same-chunk (block-diagonal) entries of
//            M_g M_g^T in fp32 for M = Z or M = V (K = the matrix's width);
//            the update-clipping norms come from these blocks.
//   kGroup   a run of consecutive groups of G chunks of one fast-weight slot,
//            each group's tiles being its apply tiles
//              O_g = Z_g W_s^T + S_g V_g            (W_s = state at group start)
//            and its update tiles
//              W <- W_s + V_g^T Z_g
//            in one launch.  The fp32 state is kept as two 16-bit planes:
//            hi, the upper half of W's bits rounded half up in magnitude (a
//            bf16 value within half an ulp of W: the apply tiles' operand),
//            and lo, the signed remainder, so (hi << 16) + lo is W's bits
//            exactly.  hi is double-buffered (the apply tiles of a group read
//            the plane that its update tiles do not write).  An update tile
//            accumulates V_g^T Z_g from zero in TMEM.  Its epilogue works in
//            64-column slices of each warp's 32 rows: TMA brings the slice's
//            block of both planes (or, at a document start, of W_0) into
//            shared memory (two slices in flight; the producer prefetched the
//            tile's block into L2 when the tile started), each thread rebuilds
//            its row's fp32 W_s there, adds the accumulator row from TMEM in
//            one fp32 rounding, writes the new planes back in place, and TMA
//            stores them.  No state byte passes through the load/store units.
//            Against a separate fp32 state and bf16 copy this writes 4 bytes
//            of state per element and group instead of 6, and the apply and
//            update tiles read the same hi plane.
//            Applying W_s to every chunk of the group plus the intra-group
//            correction S_g V_g equals applying each chunk's own pre-update
//            state (the deltas are additive, appendix B of the "In-Place
//            Test-Time Training" summary page).
//            Groups follow one another inside the launch through completion
//            counters in global memory, one per (group, 256-row block of W):
//            an apply tile of group j waits, before it loads W_s, until every
//            update tile of group j-1 for its rows has stored them; an update
//            tile of group j waits, before its epilogue touches W, until the
//            update tiles and the apply tiles of group j-1 for its rows are
//            done (its stores overwrite what they wrote and what they read).
//            Tiles are claimed in order and wait only on earlier tiles, so
//            with every CTA resident the launch cannot deadlock; the waits are
//            bounded like every other wait of the engine.
#pragma once

#include <cuda_bf16.h>
#include <cuda.h>
#include <cstdint>

#include "sm100_ptx.cuh"

namespace ttt {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB: this CTA's 128 A rows
constexpr int kBHalfBytes = (kBN / 2) * kBK * 2;  // 16 KB: this CTA's 128 B rows
constexpr int kStageBytes = kABytes + kBHalfBytes;  // 32 KB per CTA
constexpr int kTmemCols = 2 * kBN;              // two fp32 accumulators
constexpr int kSchedRing = 4;
constexpr int kGemmThreads = 192;
constexpr int kMaxGroups = 256;
// SwiGLU raster: tile pairs (of 256 token rows) per column sweep.  One sweep
// streams all of W_gate and W_up (100 MB at the Qwen3-4B shape) while its X
// rows (32 x 256 tokens: 42 MB) stay in L2; measured against sweeps of 8, 16,
// 24 and 48 pairs, 32 gave the fastest step.
constexpr int kSwizzlePairs = 32;
constexpr uint16_t kPairMask = 0x3;  // both CTAs of the cluster
// Update-tile epilogue buffers, per epilogue warp: two slice buffers, each the
// hi and the lo plane of a 32-row x 64-column block of W as TMA lays out a box
// with 128-byte swizzle (16-byte chunk q of row r at q ^ (r % 8)).
constexpr int kEpiBoxBytes = 32 * 128;              // one plane of one slice
constexpr int kEpiBufBytes = 2 * kEpiBoxBytes;      // hi, then lo
constexpr int kEpiBytesPerWarp = 2 * kEpiBufBytes;  // two slices in flight
constexpr int kEpiWarps = 4;

enum GemmMode : int { kSwiGLU = 0, kLinear = 1, kSGram = 2, kGroup = 3, kDGram = 4 };

// Tensor-map slots per mode (B boxes are the half that one CTA of a pair holds).
//   kSwiGLU: 0 X (box 64x128), 1 Wg (64x128), 2 Wu (64x128)
//   kLinear: 0 A (64x128), 1 B (64x128)
//   kSGram:  0 Z (64x128), 1 Z (64x128)
//   kDGram:  0 Z or V (64x128), 1 the same (64x128); `f` holds its width
//   kGroup:  0 Z (64x128), 1 hi[0] of the slot (64x128), 2 S (64x128),
//            3 V MN-major (64x64), 4 V MN-major with the run's K extent,
//            5 Z MN-major (64x64) with the run's K extent,
//            6 lo of the slot (64x128, L2-prefetch boxes), 7 hi[1] (64x128),
//            8 W_0 bf16 (64x128); the update epilogue's 64x32 boxes:
//            9 hi[0], 10 hi[1], 11 lo, 12 W_0
constexpr int kNumMaps = 13;

// kGroup per-group flags
constexpr uint8_t kGrpReset = 1;  // document start: the group's state is W_0
constexpr uint8_t kGrpInWb1 = 2;  // W_s's hi plane is hi[1] (else hi[0]; ignored with kGrpReset)
constexpr uint8_t kGrpOutWb1 = 4; // the update tiles write the new hi plane to hi[1] (else hi[0])

struct GemmArgs {
  CUtensorMap map[kNumMaps];
  int n_rows;    // tokens of the call (rows of X/Z/U/V/O)
  int d, f;
  int chunk;
  float alpha;   // kLinear: the output scale (eta for the target projection)
  int kdim;      // kLinear: the K extent (d for the target projection, f for O = Z W_0^T)
  int* counter;  // dynamic tile-pair counter, zero at launch
  int* err;      // workspace error word
  void* out0;    // kSwiGLU: Z; kLinear: V or O (n_rows x d); kSGram: S; kGroup: O
  // groups
  int s_pad;         // row/column pitch of one S block (multiple of 256)
  int n_groups;      // groups of the launch (kSGram, kDGram, kGroup)
  int g_start[kMaxGroups];
  int g_len[kMaxGroups];
  // kGroup
  int g_tile[kMaxGroups + 1];  // first tile pair of each group; [n_groups] = all pairs
  uint8_t g_flags[kMaxGroups];  // kGrp* bits
  int slot0;  // S slot of the run's first group (group j uses slot0 + j)
  // completion counters, zero at launch: [0, n_groups * npd) update tiles,
  // [n_groups * npd, 2 * n_groups * npd) apply tiles, npd = ceil(d / 256);
  // each tile pair adds one per epilogue warp of both CTAs
  int* dep;
  // failure-detection test hook: the leader of the pair that claims tile 0
  // withholds that tile's first ring block, so its bounded waits run out
  int test_withhold_block;
};

struct TileInfo {
  int kind;  // 0 plain/apply, 1 update
  int m0, n0;
  int g;
  int nkb1, nkb2;  // MMA K blocks: main operands, then the intra-group correction
  bool valid;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Exclusive end (multiple of 64) of the K range of the intra-group correction
// for the 128-row tile m of a group of `len` tokens: the start of the chunk
// that holds the tile's last row, rounded up to the K block.
__device__ __forceinline__ int corr_kbound(int len, int m, int chunk) {
  int last = min(m * kBM + kBM - 1, len - 1);
  int cs = (last / chunk) * chunk;
  return cdiv(cs, kBK) * kBK;
}

// Number of tile pairs (work items of a cluster).  Pair p covers the 128-row
// blocks 2*mp and 2*mp + 1 (one per CTA) of one column block.
template <int MODE>
__device__ __forceinline__ int num_tiles(const GemmArgs& a) {
  if (MODE == kSwiGLU) return cdiv(cdiv(a.n_rows, kBM), 2) * cdiv(a.f, kBM);
  if (MODE == kLinear) return cdiv(cdiv(a.n_rows, kBM), 2) * cdiv(a.d, kBN);
  if (MODE == kSGram || MODE == kDGram)
    return a.n_groups * cdiv(cdiv(a.s_pad, kBM), 2) * cdiv(a.s_pad, kBN);
  return a.g_tile[a.n_groups];
}

// Completion-counter targets of one group (kGroup): every tile pair of the
// 256-row block adds 2 * kEpiWarps.
__device__ __forceinline__ int upd_target(const GemmArgs& a) { return 2 * kEpiWarps * cdiv(a.f, kBN); }
__device__ __forceinline__ int app_target(const GemmArgs& a, int g) {
  return 2 * kEpiWarps * cdiv(cdiv(a.g_len[g], kBM), 2);
}
__device__ __forceinline__ int* upd_counter(const GemmArgs& a, int g, int blk) {
  return a.dep + g * cdiv(a.d, kBN) + blk;
}
__device__ __forceinline__ int* app_counter(const GemmArgs& a, int g, int blk) {
  return a.dep + (a.n_groups + g) * cdiv(a.d, kBN) + blk;
}

// The tile of pair `t` that CTA `rank` computes.  Everything that decides the
// ring's block sequence (validity, block counts) depends on the pair only, so
// both CTAs stream identical B blocks in the same order.
template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int t, int rank) {
  TileInfo ti{};
  ti.valid = true;
  ti.nkb2 = 0;
  ti.kind = 0;
  ti.g = 0;
  if (MODE == kSwiGLU) {
    const int mpt = cdiv(cdiv(a.n_rows, kBM), 2), nt = cdiv(a.f, kBM);
    const int gsz = kSwizzlePairs * nt;
    const int gid = t / gsz, first = gid * kSwizzlePairs;
    const int gm = min(kSwizzlePairs, mpt - first);
    const int w = t % gsz;
    ti.m0 = (2 * (first + w % gm) + rank) * kBM;
    ti.n0 = (w / gm) * kBM;
    ti.nkb1 = cdiv(a.d, kBK);
  } else if (MODE == kLinear) {
    const int nt = cdiv(a.d, kBN);
    ti.m0 = (2 * (t / nt) + rank) * kBM;
    ti.n0 = (t % nt) * kBN;
    ti.nkb1 = cdiv(a.kdim, kBK);
  } else if (MODE == kSGram) {
    const int mpt = cdiv(cdiv(a.s_pad, kBM), 2), nt = cdiv(a.s_pad, kBN);
    const int g = t / (mpt * nt), r = t % (mpt * nt);
    const int mp = r / nt, n = r % nt;
    const int len = a.g_len[g];
    ti.g = g;
    ti.m0 = (2 * mp + rank) * kBM;
    ti.n0 = n * kBN;
    // the pair is computed if either tile is needed; the epilogue's mask makes
    // the extra entries zero
    ti.valid = (2 * mp * kBM < len) && (ti.n0 < corr_kbound(len, 2 * mp + 1, a.chunk));
    ti.nkb1 = cdiv(a.f, kBK);
  } else if (MODE == kDGram) {
    const int mpt = cdiv(cdiv(a.s_pad, kBM), 2), nt = cdiv(a.s_pad, kBN);
    const int g = t / (mpt * nt), r = t % (mpt * nt);
    const int mp = r / nt, n = r % nt;
    const int len = a.g_len[g];
    ti.g = g;
    ti.m0 = (2 * mp + rank) * kBM;
    ti.n0 = n * kBN;
    // computed when the pair's rows and the tile's columns share a chunk
    const int r0 = 2 * mp * kBM, r1 = min(r0 + 2 * kBM, len) - 1;
    const int c0 = ti.n0, c1 = min(c0 + kBN, len) - 1;
    ti.valid = (r0 < len) && (c0 < len) && (r0 / a.chunk <= c1 / a.chunk) &&
               (c0 / a.chunk <= r1 / a.chunk);
    ti.nkb1 = cdiv(a.f, kBK);
  } else {
    // the group of pair t: the last g with g_tile[g] <= t
    int g = 0;
#pragma unroll
    for (int step = kMaxGroups / 2; step > 0; step >>= 1)
      if (g + step < a.n_groups && a.g_tile[g + step] <= t) g += step;
    const int len = a.g_len[g], tt = t - a.g_tile[g];
    const int mpt = cdiv(cdiv(len, kBM), 2);
    ti.g = g;
    if (tt < mpt * cdiv(a.d, kBN)) {
      // apply tiles, column-block major: the first ones need the rows of W_s
      // that the previous group's first update tiles wrote
      const int mp = tt % mpt;
      ti.m0 = (2 * mp + rank) * kBM;
      ti.n0 = (tt / mpt) * kBN;
      ti.nkb1 = cdiv(a.f, kBK);
      // the correction range of the pair's lower tile; for its upper tile the
      // extra blocks meet S entries that the Gram kernel masked to zero
      ti.nkb2 = corr_kbound(len, 2 * mp + 1, a.chunk) / kBK;
    } else {
      const int u = tt - mpt * cdiv(a.d, kBN), ntU = cdiv(a.f, kBN);
      ti.kind = 1;
      ti.m0 = (2 * (u / ntU) + rank) * kBM;
      ti.n0 = (u % ntU) * kBN;
      ti.nkb1 = cdiv(len, kBK);
    }
  }
  return ti;
}

// Bytes that one ring block of the pair's tiles brings into both CTAs (what
// the leader's full barrier expects).
constexpr uint32_t kBlockBytesPair = 2u * kStageBytes;

// Issue this CTA's TMA loads of ring block `kb` of tile `ti` into stage
// buffers sa / sb: its A rows and its half (`rank`) of the B block, with
// completion signalled on the leader's barrier `bar` (a shared::cluster
// address).
template <int MODE>
__device__ __forceinline__ void load_kblock(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                            uint8_t* sa, uint8_t* sb, uint32_t bar) {
  const int kh = kBN / 2;  // B rows (or MN columns) per half
  if (MODE == kSwiGLU) {
    tma_load_2d_pair(sa, &a.map[0], bar, kb * kBK, ti.m0);
    tma_load_2d_pair(sb, &a.map[1 + rank], bar, kb * kBK, ti.n0);
  } else if (MODE == kLinear) {
    tma_load_2d_pair(sa, &a.map[0], bar, kb * kBK, ti.m0);
    tma_load_2d_pair(sb, &a.map[1], bar, kb * kBK, ti.n0 + rank * kh);
  } else if (MODE == kSGram || MODE == kDGram) {
    const int gs = a.g_start[ti.g];
    tma_load_2d_pair(sa, &a.map[0], bar, kb * kBK, gs + ti.m0);
    tma_load_2d_pair(sb, &a.map[1], bar, kb * kBK, gs + ti.n0 + rank * kh);
  } else {
    const int gs = a.g_start[ti.g];
    if (ti.kind == 0) {
      // the intra-group correction S_g V_g first (it does not depend on W_s),
      // then the main product Z_g W_s^T
      if (kb >= ti.nkb2) {
        const int k = (kb - ti.nkb2) * kBK;
        const uint8_t fl = a.g_flags[ti.g];
        const CUtensorMap* mb = (fl & kGrpReset) ? &a.map[8] : (fl & kGrpInWb1) ? &a.map[7] : &a.map[1];
        tma_load_2d_pair(sa, &a.map[0], bar, k, gs + ti.m0);
        tma_load_2d_pair(sb, mb, bar, k, ti.n0 + rank * kh);
      } else {
        const int k2 = kb * kBK;
        tma_load_2d_pair(sa, &a.map[2], bar, k2, (a.slot0 + ti.g) * a.s_pad + ti.m0);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          tma_load_2d_pair(sb + q * 8192, &a.map[3], bar, ti.n0 + rank * kh + q * 64, gs + k2);
      }
    } else {
      const int k = gs + kb * kBK;
#pragma unroll
      for (int q = 0; q < kBM / 64; ++q)
        tma_load_2d_pair(sa + q * 8192, &a.map[4], bar, ti.m0 + q * 64, k);
#pragma unroll
      for (int q = 0; q < 2; ++q)
        tma_load_2d_pair(sb + q * 8192, &a.map[5], bar, ti.n0 + rank * kh + q * 64, k);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// SiLU with the fast-division intrinsic (a few ulp of fp32; the result is
// rounded to bf16).
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// The two 16-bit planes of an fp32 value's bits b: hi = the upper half
// rounded half up in magnitude (a bf16 within half an ulp of the value; b +
// 0x8000 cannot carry into the sign for a finite value), lo = b - (hi << 16)
// as a signed 16-bit remainder, in [-0x8000, 0x7fff].  join_hi_lo inverts
// them exactly (the low 16 bits of its arguments are used).
__device__ __forceinline__ uint32_t hi_of(uint32_t b) { return (b + 0x8000u) >> 16; }
__device__ __forceinline__ uint32_t lo_of(uint32_t b, uint32_t h) { return (b - (h << 16)) & 0xFFFFu; }
__device__ __forceinline__ uint32_t join_hi_lo(uint32_t h, uint32_t l) {
  return ((h & 0xFFFFu) << 16) + static_cast<uint32_t>(static_cast<int32_t>(static_cast<int16_t>(l & 0xFFFFu)));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr)
               : "memory");
}

// Store 32 consecutive bf16 values (packed in 16 words) if the 8-groups are in range.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const uint32_t (&p)[16],
                                              int cols_left) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < cols_left) {
      uint4 v = make_uint4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
      *reinterpret_cast<uint4*>(dst + q * 8) = v;
    }
  }
}

template <int MODE>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, const TileInfo& ti,
                                              uint32_t tacc, int row) {
  uint32_t r[32];
  if (MODE == kSwiGLU) {
    const int grow = ti.m0 + row;
    __nv_bfloat16* zrow = reinterpret_cast<__nv_bfloat16*>(a.out0) + (size_t)grow * a.f;
#pragma unroll 1
    for (int s = 0; s < kBM / 32; ++s) {
      uint32_t u[32];
      tmem_ld32(tacc + s * 32, r);
      tmem_ld_wait(r);
      tmem_ld32(tacc + kBM + s * 32, u);
      tmem_ld_wait(u);
      uint32_t p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float z0 = silu_f(__uint_as_float(r[2 * j])) * __uint_as_float(u[2 * j]);
        float z1 = silu_f(__uint_as_float(r[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
        p[j] = pack_bf16x2(z0, z1);
      }
      const int col = ti.n0 + s * 32;
      if (grow < a.n_rows) store_bf16x32(zrow + col, p, a.f - col);
    }
  } else if (MODE == kLinear || MODE == kGroup) {
    // plain bf16 store of alpha * acc (kLinear) or acc (the apply tiles of
    // kGroup; its update tiles have their own epilogue, update_epilogue)
    const float alpha = (MODE == kLinear) ? a.alpha : 1.0f;
    const int grow = (MODE == kLinear) ? ti.m0 + row : a.g_start[ti.g] + ti.m0 + row;
    const bool ok = (MODE == kLinear) ? (grow < a.n_rows) : (ti.m0 + row < a.g_len[ti.g]);
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out0) + (size_t)grow * a.d;
#pragma unroll 1
    for (int s = 0; s < kBN / 32; ++s) {
      tmem_ld32(tacc + s * 32, r);
      tmem_ld_wait(r);
      uint32_t p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        p[j] = pack_bf16x2(alpha * __uint_as_float(r[2 * j]),
                           alpha * __uint_as_float(r[2 * j + 1]));
      const int col = ti.n0 + s * 32;
      if (ok) store_bf16x32(orow + col, p, a.d - col);
    }
  } else if (MODE == kDGram) {
    // same-chunk entries of the Gram block in fp32, everything else 0
    const int len = a.g_len[ti.g];
    const int i = ti.m0 + row;
    // kept: row i in the group, column j in row i's chunk
    const int jlo = (i / a.chunk) * a.chunk;
    const int jhi = i < len ? min(len, jlo + a.chunk) : 0;
    float* grow = reinterpret_cast<float*>(a.out0) + ((size_t)ti.g * a.s_pad + i) * a.s_pad;
#pragma unroll 1
    for (int s = 0; s < kBN / 32; ++s) {
      tmem_ld32(tacc + s * 32, r);
      tmem_ld_wait(r);
      const int j0 = ti.n0 + s * 32;
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const bool keep = j0 + j >= jlo && j0 + j < jhi;
        v[j] = keep ? __uint_as_float(r[j]) : 0.0f;
      }
      if (i < a.s_pad) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(grow + j0 + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  } else {  // kSGram
    const int len = a.g_len[ti.g];
    const int i = ti.m0 + row;
    // kept: row i in the group, column j in a chunk strictly before row i's
    // (one division per row, none per entry)
    const int jend = i < len ? min(len, (i / a.chunk) * a.chunk) : 0;
    __nv_bfloat16* srow =
        reinterpret_cast<__nv_bfloat16*>(a.out0) + ((size_t)ti.g * a.s_pad + i) * a.s_pad;
#pragma unroll 1
    for (int s = 0; s < kBN / 32; ++s) {
      tmem_ld32(tacc + s * 32, r);
      tmem_ld_wait(r);
      const int j0 = ti.n0 + s * 32;
      uint32_t p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int ja = j0 + 2 * j;
        const bool ka = ja < jend, kb = ja + 1 < jend;
        p[j] = pack_bf16x2(ka ? __uint_as_float(r[2 * j]) : 0.0f,
                           kb ? __uint_as_float(r[2 * j + 1]) : 0.0f);
      }
      if (i < a.s_pad) store_bf16x32(srow + j0, p, a.s_pad - j0);
    }
  }
}

// The update tiles' epilogue state of one epilogue warp: its two slice
// buffers (`buf`, kEpiBytesPerWarp bytes, 1024-byte aligned), their TMA
// barriers, the barriers' phase bits and which buffers have a load in flight.
struct SliceBuffers {
  uint8_t* buf;
  uint64_t* bar;  // [2]
  uint32_t phase;
  uint32_t pending;
};

// The maps the update epilogue of group g reads its state from and writes it to.
__device__ __forceinline__ const CUtensorMap* upd_hi_in(const GemmArgs& a, int g) {
  const uint8_t fl = a.g_flags[g];
  return (fl & kGrpReset) ? &a.map[12] : (fl & kGrpInWb1) ? &a.map[10] : &a.map[9];
}
__device__ __forceinline__ const CUtensorMap* upd_hi_out(const GemmArgs& a, int g) {
  return (a.g_flags[g] & kGrpOutWb1) ? &a.map[10] : &a.map[9];
}

// Whether slice u of this warp's rows holds any element of W (d x f): a
// slice wholly outside (a tile past a d or f that is not a multiple of 256)
// is neither loaded nor stored.
__device__ __forceinline__ bool upd_slice_live(const GemmArgs& a, const TileInfo& ti, int sub, int u) {
  return ti.m0 + sub * 32 < a.d && ti.n0 + u * 64 < a.f;
}

// Lane 0: start the TMA loads of slice u (64 columns) of this warp's 32 rows of
// W_s into buffer b: the hi plane (W_0's bf16 values at a document start) and
// the lo plane (none at a document start: it is zero there).  A dead slice
// completes the barrier's phase with no bytes.
__device__ __forceinline__ void upd_load_slice(const GemmArgs& a, const TileInfo& ti, int sub, int u,
                                               int b, SliceBuffers& sb) {
  const bool from_w0 = a.g_flags[ti.g] & kGrpReset;
  const bool live = upd_slice_live(a, ti, sub, u);
  uint8_t* dst = sb.buf + b * kEpiBufBytes;
  const uint32_t bar = smem_u32(&sb.bar[b]);
  const int c0 = ti.n0 + u * 64, r0 = ti.m0 + sub * 32;
  mbar_arrive_expect_tx(&sb.bar[b], !live ? 0 : from_w0 ? kEpiBoxBytes : kEpiBufBytes);
  if (!live) return;
  tma_load_2d_pair(dst, upd_hi_in(a, ti.g), bar, c0, r0);
  if (!from_w0) tma_load_2d_pair(dst + kEpiBoxBytes, &a.map[11], bar, c0, r0);
}

// Fast-weight update of one update tile, for one epilogue warp (its 32 rows,
// one per lane): W <- W_s + acc in one fp32 rounding, in four 64-column
// slices.  The loads of slices 0 and 1 were started before the accumulator
// was ready (upd_load_slice).  Per slice: wait for its state block, take the
// accumulator row from TMEM, rebuild W_s from the planes in shared memory,
// add, write the new planes over the old ones, and TMA-store them (the hi
// plane to the group's output plane, lo in place); the buffer then takes
// slice u + 2.  The global writes complete in the caller (bulk_wait_group).
// Returns false if a wait ran out.
__device__ __forceinline__ bool update_epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                                int sub, int lane, SliceBuffers& sb,
                                                volatile int* abort_flag) {
  const bool from_w0 = a.g_flags[ti.g] & kGrpReset;
  const CUtensorMap* m_out = upd_hi_out(a, ti.g);
  const int r0 = ti.m0 + sub * 32;
  uint32_t r[32], v[32];
#pragma unroll 1
  for (int u = 0; u < kBN / 64; ++u) {
    const int b = u & 1;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sb.bar[b], (sb.phase >> b) & 1u, abort_flag, a.err, kErrWaitEpi);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    sb.phase ^= 1u << b;
    sb.pending &= ~(1u << b);
    tmem_ld32(tacc + u * 64, r);
    tmem_ld_wait(r);
    tmem_ld32(tacc + u * 64 + 32, v);
    tmem_ld_wait(v);
    // this lane's row of the slice: 8 chunks of 8 columns per plane
    const uint32_t hrow = smem_u32(sb.buf + b * kEpiBufBytes) + lane * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t off = static_cast<uint32_t>((q ^ (lane & 7)) << 4);
      uint32_t hw[4], lw[4] = {0u, 0u, 0u, 0u};
      ld_shared_v4(hrow + off, hw);
      if (!from_w0) ld_shared_v4(hrow + kEpiBoxBytes + off, lw);
      uint32_t ho[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t d0 = q < 4 ? r[8 * q + 2 * e] : v[8 * (q - 4) + 2 * e];
        const uint32_t d1 = q < 4 ? r[8 * q + 2 * e + 1] : v[8 * (q - 4) + 2 * e + 1];
        const uint32_t b0 = __float_as_uint(__uint_as_float(join_hi_lo(hw[e], lw[e])) + __uint_as_float(d0));
        const uint32_t b1 =
            __float_as_uint(__uint_as_float(join_hi_lo(hw[e] >> 16, lw[e] >> 16)) + __uint_as_float(d1));
        const uint32_t h0 = hi_of(b0), h1 = hi_of(b1);
        ho[e] = h0 | (h1 << 16);
        lo[e] = lo_of(b0, h0) | (lo_of(b1, h1) << 16);
      }
      st_shared_v4(hrow + off, ho[0], ho[1], ho[2], ho[3]);
      st_shared_v4(hrow + kEpiBoxBytes + off, lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      uint8_t* src = sb.buf + b * kEpiBufBytes;
      if (upd_slice_live(a, ti, sub, u)) {
        tma_store_2d(m_out, src, ti.n0 + u * 64, r0);
        tma_store_2d(&a.map[11], src + kEpiBoxBytes, ti.n0 + u * 64, r0);
      }
      bulk_commit_group();
      if (u + 2 < kBN / 64) {
        bulk_wait_group_read<0>();  // the stores have read the buffer
        upd_load_slice(a, ti, sub, u + 2, b, sb);
      }
    }
    if (u + 2 < kBN / 64) sb.pending |= 1u << b;
    __syncwarp();
  }
  return true;
}

// Ring depth and dynamic shared memory of each mode.
template <int MODE>
__host__ __device__ constexpr int stages_of() {
  return MODE == kGroup ? 5 : 7;
}
template <int MODE>
__host__ __device__ constexpr int smem_bytes_of() {
  return 1024 /*align*/ + stages_of<MODE>() * kStageBytes + 1024 /*barriers*/ +
         (MODE == kGroup ? kEpiWarps * kEpiBytesPerWarp : 0);
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) tc_gemm_kernel(const __grid_constant__ GemmArgs a) {
  constexpr int kStages = stages_of<MODE>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the dynamic window starts at the same offset in every CTA, so aligning the
  // same way keeps the layout (MMA operand halves, barriers) identical in both
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;                       // [kStages]  (used in the leader)
  uint64_t* empty = full + kStages;            // [kStages]
  uint64_t* acc_full = empty + kStages;        // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2]        (used in the leader)
  uint64_t* sched_full = acc_empty + 2;        // [kSchedRing]
  uint64_t* sched_empty = sched_full + kSchedRing;  // [kSchedRing] (used in the leader)
  uint64_t* drain = sched_empty + kSchedRing;  // [1]
  uint64_t* epi_bar = drain + 1;               // [kEpiWarps][2] (update-tile state loads)
  int* sched_item = reinterpret_cast<int*>(epi_bar + 2 * kEpiWarps);  // [kSchedRing]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sched_item + kSchedRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [kEpiWarps][kEpiBytesPerWarp], 1024-byte aligned (128-byte swizzle boxes)
  uint8_t* epi_smem = smem + kStages * kStageBytes + 1024;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int ntiles = num_tiles<MODE>(a);
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;

  // Arrive on the leader's copy of a barrier (local in the leader, remote in the peer).
  auto arrive_leader = [&](uint64_t* bar) {
    if (leader)
      mbar_arrive(bar);
    else
      mbar_arrive_cluster(cluster_map(smem_u32(bar), 0));
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);   // the leader's expect; both CTAs' bytes
      mbar_init(&empty[s], 1);  // the leader's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kEpiWarps);  // both CTAs' epilogue warps
    }
    for (int s = 0; s < kSchedRing; ++s) {
      mbar_init(&sched_full[s], 1);
      // leader: its MMA + epilogue warps, and the peer's producer + epilogue warps
      mbar_init(&sched_empty[s], 2 + 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(&epi_bar[b], 1);  // the loading lane's expect
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and TMEM exist before any pair traffic
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above may overlap the previous kernel's tail (programmatic
  // dependent launch); no global memory is touched before that kernel is done.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (+ the pair's tile scheduler on the leader)
#pragma unroll 1
      for (int q = 0; q < (MODE == kGroup ? kNumMaps : 3); ++q) tma_prefetch_desc(&a.map[q]);
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      bool ok = true;
#pragma unroll 1
      for (int it = 0; ok; ++it) {
        const int slot = it % kSchedRing;
        const uint32_t sp = (it / kSchedRing) & 1;
        int t;
        if (leader) {
          if (!mbar_wait(&sched_empty[slot], sp ^ 1, abort_flag, a.err, kErrWaitSched)) break;
          t = atomicAdd(a.counter, 1);
          sched_item[slot] = t;
          st_cluster_u32(cluster_map(smem_u32(&sched_item[slot]), 1), static_cast<uint32_t>(t));
          mbar_arrive(&sched_full[slot]);
          mbar_arrive_cluster(cluster_map(smem_u32(&sched_full[slot]), 1));
        } else {
          if (!mbar_wait(&sched_full[slot], sp, abort_flag, a.err, kErrWaitSched)) break;
          t = sched_item[slot];
          arrive_leader(&sched_empty[slot]);
        }
        if (t >= ntiles) break;
        const TileInfo ti = decode_tile<MODE>(a, t, rank);
        if (!ti.valid) continue;
        if (MODE == kGroup && ti.kind == 1 && !(a.g_flags[ti.g] & kGrpReset)) {
          // the epilogue adds this tile's block of W_s (both planes) after
          // the MMAs; bring it into L2 now so those reads hit there (L2 is the
          // point of coherence, so a prefetch ahead of the block's last
          // writer is safe)
          const CUtensorMap* mhi = (a.g_flags[ti.g] & kGrpInWb1) ? &a.map[7] : &a.map[1];
          for (int b = 0; b < kBN / kBK; ++b) {
            tma_prefetch_l2_2d(mhi, ti.n0 + b * kBK, ti.m0);
            tma_prefetch_l2_2d(&a.map[6], ti.n0 + b * kBK, ti.m0);
          }
        }
        const int nkb = ti.nkb1 + ti.nkb2;
#pragma unroll 1
        for (int kb = 0; kb < nkb; ++kb) {
          if (MODE == kGroup && ti.kind == 0 && kb == ti.nkb2 && ti.g > 0 &&
              !(a.g_flags[ti.g] & kGrpReset)) {
            // W_s rows [n0, n0 + 256) come from the previous group's update
            // tiles of this launch
            if (!dep_wait(upd_counter(a, ti.g - 1, ti.n0 / kBN), upd_target(a), abort_flag, a.err,
                          kErrWaitDep)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();  // their generic stores before our TMA reads
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err, kErrWaitSmemEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = stage_base + stage * kStageBytes;
          if (leader) mbar_arrive_expect_tx(&full[stage], kBlockBytesPair);
          if (!(a.test_withhold_block && leader && t == 0 && kb == 0))
            load_kblock<MODE>(a, ti, kb, rank, sa, sa + kABytes, cluster_map(smem_u32(&full[stage]), 0));
          ++fills;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (*abort_flag && leader) {
        // let every load still in flight land before the CTA's smem is released
        for (int s = 0; s < kStages && s < fills; ++s) {
          const uint32_t p = (s < stage) ? phase : (phase ^ 1);
          volatile int never = 0;
          mbar_wait(&full[s], p, &never, a.err, kErrWaitDrain);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer for the pair
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t sa_base = smem_u32(stage_base);
      uint32_t sa_cur = sa_base;  // shared address of ring stage `stage`
      int acc_it = 0;
      bool ok = true;
#pragma unroll 1
      for (int it = 0; ok; ++it) {
        const int slot = it % kSchedRing;
        if (!mbar_wait(&sched_full[slot], (it / kSchedRing) & 1, abort_flag, a.err,
                       kErrWaitSched))
          break;
        const int t = sched_item[slot];
        mbar_arrive(&sched_empty[slot]);
        if (t >= ntiles) break;
        const TileInfo ti = decode_tile<MODE>(a, t, rank);
        if (!ti.valid) continue;
        const int buf = acc_it & 1;
        if (!mbar_wait(&acc_empty[buf], ((acc_it >> 1) & 1) ^ 1, abort_flag, a.err,
                       kErrWaitAccEmpty))
          break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + buf * kBN;
        // A tile's ring blocks come in up to two segments of fixed operand
        // layout: the main K loop and the intra-group correction.  This one thread must keep up with the
        // tensor pipe (4 MMAs of 128 cycles per block), so everything that
        // depends only on the segment is hoisted: a block costs a wait, two
        // ORs, four MMAs with one add each, and a commit.
        constexpr uint64_t kK = sdesc_sw128_hi(0, 1024), kMN = sdesc_sw128_hi(8192, 1024);
        // apply tiles: correction first, then the main product
        const bool apply = MODE == kGroup && ti.kind == 0;
        uint32_t accum = 0u;
#pragma unroll 1
        for (int seg = 0; seg < 2 && ok; ++seg) {
          const int cnt = apply ? (seg == 0 ? ti.nkb2 : ti.nkb1) : (seg == 0 ? ti.nkb1 : 0);
          // operand majors: 0 both K-major, 1 B MN-major (correction),
          // 2 both MN-major (update)
          const int lay = apply ? (seg == 0 ? 1 : 0) : ((MODE == kGroup && ti.kind == 1) ? 2 : 0);
          const uint32_t idesc = lay == 0   ? idesc_bf16_f32(2 * kBM, kBN, false, false)
                                 : lay == 1 ? idesc_bf16_f32(2 * kBM, kBN, false, true)
                                            : idesc_bf16_f32(2 * kBM, kBN, true, true);
          const uint64_t ahi = lay == 2 ? kMN : kK, bhi = lay >= 1 ? kMN : kK;
          const uint32_t astep = lay == 2 ? (2048 >> 4) : (32 >> 4);
          const uint32_t bstep = lay >= 1 ? (2048 >> 4) : (32 >> 4);
#pragma unroll 1
          for (int i = 0; i < cnt; ++i) {
            if (!mbar_wait(&full[stage], phase, abort_flag, a.err, kErrWaitTmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint64_t ad = ahi | ((sa_cur & 0x3FFFFu) >> 4);
            uint64_t bd = bhi | (((sa_cur + kABytes) & 0x3FFFFu) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              tc_mma_bf16_pair(tacc, ad, bd, idesc, accum);
              accum = 1u;
              ad += astep;
              bd += bstep;
            }
            // the stage is free in both CTAs once the pair's MMAs have read it
            tc_commit_pair_mc(&empty[stage], kPairMask);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
              sa_cur = sa_base;
            } else {
              sa_cur += kStageBytes;
            }
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&acc_full[buf], kPairMask);
        ++acc_it;
      }
      // every tcgen05 op of the pair (and the arrivals it signals) completes
      // before the pair leaves
      tc_commit_pair(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, a.err, kErrWaitDrain);
    }
  } else {
    // ---------------- epilogue warps
    const int sub = warp & 3;  // TMEM sub-partition this warp may access
    const int row = sub * 32 + lane;
    SliceBuffers sb{epi_smem + (warp - 2) * kEpiBytesPerWarp, epi_bar + (warp - 2) * 2, 0u, 0u};
    int acc_it = 0;
#pragma unroll 1
    for (int it = 0;; ++it) {
      // lane 0 waits; the result is broadcast so the warp stays converged for
      // the .sync.aligned TMEM loads
      const int slot = it % kSchedRing;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(&sched_full[slot], (it / kSchedRing) & 1, abort_flag, a.err, kErrWaitSched);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int t = sched_item[slot];
      __syncwarp();
      if (lane == 0) arrive_leader(&sched_empty[slot]);
      if (t >= ntiles) break;
      const TileInfo ti = decode_tile<MODE>(a, t, rank);
      if (!ti.valid) continue;
      const bool upd = MODE == kGroup && ti.kind == 1;
      if (upd) {
        if (ti.g > 0) {
          // this tile rewrites the lo block that the previous group's update
          // tile wrote and the hi rows that its apply tiles read
          const int blk = ti.m0 / kBN;
          int okd = 1;
          if (lane == 0) {
            okd = dep_wait(upd_counter(a, ti.g - 1, blk), upd_target(a), abort_flag, a.err, kErrWaitDep);
            if (okd)
              okd = dep_wait(app_counter(a, ti.g - 1, blk), app_target(a, ti.g - 1), abort_flag, a.err,
                             kErrWaitDep);
            fence_proxy_async_global();  // their writes before our TMA reads
          }
          if (!__shfl_sync(0xffffffffu, okd, 0)) break;
        }
        // the state of the first two slices streams in while the MMAs finish
        if (lane == 0) {
          upd_load_slice(a, ti, sub, 0, 0, sb);
          upd_load_slice(a, ti, sub, 1, 1, sb);
        }
        sb.pending = 3u;
      }
      const int buf = acc_it & 1;
      if (lane == 0)
        ok = mbar_wait(&acc_full[buf], (acc_it >> 1) & 1, abort_flag, a.err, kErrWaitAccFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + buf * kBN;
      if (upd) {
        const bool okw = update_epilogue(a, ti, tacc, sub, lane, sb, abort_flag);
        // the accumulator is read (or abandoned): hand it back first
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&acc_empty[buf]);
        if (!okw) break;
        if (lane == 0) {
          // the new planes are in global memory before the next group's
          // tiles are told (they read them through TMA)
          bulk_wait_group<0>();
          fence_proxy_async_global();
          __threadfence();
          dep_signal(upd_counter(a, ti.g, ti.m0 / kBN), 1);
        }
        __syncwarp();
      } else {
        epilogue_tile<MODE>(a, ti, tacc, row);
        if (MODE == kGroup) {
          __syncwarp();
          if (lane == 0) dep_signal(app_counter(a, ti.g, ti.n0 / kBN), 1);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&acc_empty[buf]);
      }
      ++acc_it;
    }
    if (MODE == kGroup && lane == 0) {
      // before the CTA's shared memory is released: state loads still in
      // flight land, and the stores have read their buffers
      volatile int never = 0;
      for (int b2 = 0; b2 < 2; ++b2)
        if (sb.pending & (1u << b2)) mbar_wait(&sb.bar[b2], (sb.phase >> b2) & 1u, &never, a.err, kErrWaitDrain);
      bulk_wait_group<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no pair traffic targets a CTA that has left
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

static_assert(smem_bytes_of<kSwiGLU>() <= 232448 && smem_bytes_of<kGroup>() <= 232448,
              "exceeds the opt-in shared memory of one CTA");

}  // namespace ttt
