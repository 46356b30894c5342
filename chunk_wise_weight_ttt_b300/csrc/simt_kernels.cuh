// Plain CUDA-core kernels: the fp32 (FFMA) layer path, the chunk-local
// Conv1D target source, state copies and conversions, and the residual-stack
// glue.  The fp32 path computes every contraction in fp32 with no TF32.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace ttt {

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr int kMaxSpans = 256;

// 8 consecutive elements (16-byte aligned for bf16, 32-byte for fp32) as floats.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
  *reinterpret_cast<uint4*>(p) = q;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Token spans whose chunking is regular: span i covers [start[i], start[i] +
// len[i]) and its chunks are [start + c*chunk, ...) clipped to the span end.
struct SpanList {
  int n;
  int chunk;
  int start[kMaxSpans];
  int len[kMaxSpans];
};

// U[t] = sum_{j<k} conv[j] (.) X0[t + off(j)] with every term outside t's
// chunk dropped (chunk-local depthwise Conv1D); off(j) = 1 + j (next-token
// window), j (current-token window) or 1 - j (causal window), by `mode`.
// A CTA (256 threads) computes conv_tokens<TIn>() consecutive tokens x
// kConvCh channels of the tokens covered by `spans`: it stages the X0 rows
// those tokens read (tokens + KT - 1 rows) in shared memory with asynchronous
// 16-byte copies (all in flight at once; zero-filled outside the spans), so
// every row comes from HBM once.  A thread then owns 4 channels and a run of
// consecutive tokens: it keeps its KT tap weights and a window of the last KT
// rows in registers and slides the window one row per token, so shared
// memory delivers each row to it once rather than once per tap (the per-tap
// form was bound by shared-memory bandwidth).  Tokens outside every span are
// untouched.  KT = k, the number of taps (1..8).
// Grid: (ceil(span tokens / conv_tokens<TIn>()), ceil(d / kConvCh)).
constexpr int kConvCh = 256;
template <typename TIn>
__host__ __device__ constexpr int conv_tokens() { return sizeof(TIn) == 2 ? 64 : 32; }

// 16-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src), "r"(src_bytes)
               : "memory");
}

// 4 consecutive elements (8-byte aligned for bf16, 16-byte for fp32) as floats.
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 q;
  *reinterpret_cast<__nv_bfloat162*>(&q.x) = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162*>(&q.y) = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = q;
}
__device__ __forceinline__ void store4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

template <typename TIn, typename TOut, int KT>
__global__ void __launch_bounds__(256, 2) conv_target_kernel(const TIn* __restrict__ x0,
                                                          const TIn* __restrict__ conv_w,
                                                          TOut* __restrict__ u, int d,
                                                          const SpanList spans, int mode) {
  constexpr int kConvTok = conv_tokens<TIn>();
  constexpr int kRows = kConvTok + KT - 1;  // X0 rows the CTA's tokens read
  __shared__ __align__(16) TIn slab[kRows * kConvCh];
  const int first = spans.start[0];
  const int last = spans.start[spans.n - 1] + spans.len[spans.n - 1];  // exclusive
  const int t0 = first + blockIdx.x * kConvTok;
  const int ch0 = blockIdx.y * kConvCh;
  const int omin = (mode == 2) ? 2 - KT : (mode == 1 ? 0 : 1);  // smallest tap offset
  constexpr int kChunks = kConvCh / 8;                 // groups of 8 channels per row
  constexpr int kPieces = 8 * (int)sizeof(TIn) / 16;   // 16-byte copies per group
  for (int q = threadIdx.x; q < kRows * kChunks * kPieces; q += blockDim.x) {
    const int pc = q % kPieces, rc = q / kPieces;
    const int r = rc / kChunks, cg = rc % kChunks;
    const int row = t0 + omin + r, ch = ch0 + cg * 8;
    const bool in = row >= first && row < last && ch < d;
    const TIn* src = in ? x0 + (size_t)row * d + ch : x0;
    cp_async16(slab + r * kConvCh + cg * 8 + pc * (16 / (int)sizeof(TIn)),
               reinterpret_cast<const uint8_t*>(src) + pc * 16, in ? 16 : 0);
  }
  constexpr int kQuads = kConvCh / 4;     // threads per token lane (4 channels each)
  constexpr int kLanes = 256 / kQuads;    // token lanes
  constexpr int kRun = kConvTok / kLanes; // consecutive tokens per thread
  const int cq = threadIdx.x % kQuads, tl = threadIdx.x / kQuads;
  const int ch = ch0 + cq * 4;
  // window slot s holds row t + omin + s; its tap is j = s, or KT - 1 - s for
  // the causal window (off(j) = 1 - j)
  float w[KT][4];
  if (ch < d) {
#pragma unroll
    for (int s = 0; s < KT; ++s) load4(conv_w + (size_t)(mode == 2 ? KT - 1 - s : s) * d + ch, w[s]);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (ch >= d) return;
  const int r0 = tl * kRun;  // slab row of slot 0 for the thread's first token
  float win[KT][4];
#pragma unroll
  for (int s = 1; s < KT; ++s) load4(slab + (r0 + s - 1) * kConvCh + cq * 4, win[s]);
  int s_end = -1, cbeg = 0, cend = 0;  // current span end and chunk
#pragma unroll
  for (int i = 0; i < kRun; ++i) {
#pragma unroll
    for (int s = 0; s + 1 < KT; ++s)
#pragma unroll
      for (int c = 0; c < 4; ++c) win[s][c] = win[s + 1][c];
    load4(slab + (r0 + i + KT - 1) * kConvCh + cq * 4, win[KT - 1]);
    const int t = t0 + r0 + i;
    if (t >= last) continue;
    if (t >= s_end) {
      int lo = 0, hi = spans.n - 1;
      while (lo < hi) {  // last span starting at or before t
        const int mid = (lo + hi + 1) / 2;
        if (spans.start[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int s0 = spans.start[lo];
      s_end = s0 + spans.len[lo];
      if (t >= s_end) {  // in a gap between spans
        s_end = -1;
        continue;
      }
      cbeg = s0 + ((t - s0) / spans.chunk) * spans.chunk;
      cend = min(cbeg + spans.chunk, s_end);
    } else if (t >= cend) {  // the next chunk of the span
      cbeg = cend;
      cend = min(cbeg + spans.chunk, s_end);
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int s = 0; s < KT; ++s) {
      const int r = t + omin + s;
      if (r >= cbeg && r < cend) {
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaf(w[s][c], win[s][c], acc[c]);
      }
    }
    store4(u + (size_t)t * d + ch, acc);
  }
}

// Launch conv_target_kernel for k taps (1..8) on `st`.
template <typename TIn, typename TOut>
inline cudaError_t launch_conv(dim3 grid, cudaStream_t st, const TIn* x0, const TIn* conv_w, TOut* u,
                               int d, int k, const SpanList& spans, int mode) {
  using Fn = void (*)(const TIn*, const TIn*, TOut*, int, const SpanList, int);
  const Fn fns[8] = {conv_target_kernel<TIn, TOut, 1>, conv_target_kernel<TIn, TOut, 2>,
                     conv_target_kernel<TIn, TOut, 3>, conv_target_kernel<TIn, TOut, 4>,
                     conv_target_kernel<TIn, TOut, 5>, conv_target_kernel<TIn, TOut, 6>,
                     conv_target_kernel<TIn, TOut, 7>, conv_target_kernel<TIn, TOut, 8>};
  if (k < 1 || k > 8) return cudaErrorInvalidValue;
  fns[k - 1]<<<grid, 256, 0, st>>>(x0, conv_w, u, d, spans, mode);
  return cudaGetLastError();
}

// C(m,n) = alpha * sum_k A(m,k) B(k,n) + beta * C(m,n), fp32 accumulation.
// A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn], C(m,n) = C[m*ldc + n].
// 64x64 tiles, 256 threads, 4x4 outputs per thread, K staged 16 at a time.
template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) simt_gemm_kernel(int M, int N, int K, const TA* __restrict__ A,
                                                        long long sam, long long sak,
                                                        const TB* __restrict__ B, long long sbk,
                                                        long long sbn, TC* C, long long ldc,
                                                        float alpha, float beta) {
  __shared__ float As[16][64 + 1];
  __shared__ float Bs[16][64 + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i / 64, mm = i % 64;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? to_f(A[(long long)m * sam + (long long)k * sak]) : 0.0f;
      const int n = n0 + mm;
      Bs[kk][mm] = (n < N && k < K) ? to_f(B[(long long)k * sbk + (long long)n * sbn]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      TC* p = C + (long long)m * ldc + n;
      float v = alpha * acc[i][j];
      if (beta != 0.0f) v += beta * to_f(*p);
      *p = from_f<TC>(v);
    }
  }
}

// Z(m,n) = SiLU(sum_k X(m,k) Wg(n,k)) * sum_k X(m,k) Wu(n,k); X: M x K, Wg/Wu: N x K.
template <typename T>
__global__ void __launch_bounds__(256) simt_swiglu_kernel(int M, int N, int K, const T* __restrict__ X,
                                                          const T* __restrict__ Wg,
                                                          const T* __restrict__ Wu,
                                                          float* __restrict__ Z) {
  __shared__ float Xs[16][64 + 1];
  __shared__ float Gs[16][64 + 1];
  __shared__ float Us[16][64 + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float ag[4][4] = {}, au[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i % 16, rr = i / 16;
      const int k = k0 + kk;
      const int m = m0 + rr, n = n0 + rr;
      Xs[kk][rr] = (m < M && k < K) ? to_f(X[(long long)m * K + k]) : 0.0f;
      Gs[kk][rr] = (n < N && k < K) ? to_f(Wg[(long long)n * K + k]) : 0.0f;
      Us[kk][rr] = (n < N && k < K) ? to_f(Wu[(long long)n * K + k]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], g[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Xs[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        g[j] = Gs[kk][tx + 16 * j];
        u[j] = Us[kk][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag[i][j] = fmaf(a[i], g[j], ag[i][j]);
          au[i][j] = fmaf(a[i], u[j], au[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      const float g = ag[i][j];
      Z[(long long)m * N + n] = (g / (1.0f + expf(-g))) * au[i][j];
    }
  }
}

constexpr int kMaxClipGroups = 256;

// Groups of chunks whose same-chunk Gram blocks sit in `pitch` x `pitch` fp32
// blocks (one per group, in order): group i covers tokens [start[i],
// start[i] + len[i]) in chunks of `chunk` (the last may be short), at most G
// chunks per group.
struct GroupList {
  int n, chunk, G, pitch;
  int start[kMaxClipGroups];
  int len[kMaxClipGroups];
};

// Per-chunk update clipping: one 256-thread block per chunk computes
// ||V_c^T Z_c||_F^2 = sum_{i,j in c} (Z Z^T)_{ij} (V V^T)_{ij} from the Gram
// blocks (fp64 accumulation in a fixed order), and when the norm exceeds tau
// scales the chunk's rows of V (the eta-scaled target) by tau / norm, which
// scales the chunk's delta V_c^T Z_c by the same factor.
template <typename TV>
__global__ void __launch_bounds__(256) clip_scale_kernel(const float* __restrict__ gz,
                                                         const float* __restrict__ gv, TV* v,
                                                         int d, float tau, const GroupList gl) {
  const int gi = blockIdx.x / gl.G, ci = blockIdx.x % gl.G;
  if (gi >= gl.n) return;
  const int r0 = ci * gl.chunk;
  const int len = gl.len[gi];
  if (r0 >= len) return;
  const int n = min(gl.chunk, len - r0);
  const size_t base = (size_t)gi * gl.pitch * gl.pitch;
  double acc = 0.0;
  for (long long idx = threadIdx.x; idx < (long long)n * n; idx += blockDim.x) {
    const int i = r0 + (int)(idx / n), j = r0 + (int)(idx % n);
    const size_t o = base + (size_t)i * gl.pitch + j;
    acc += (double)gz[o] * (double)gv[o];
  }
  __shared__ double red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const double nrm = sqrt(fmax(red[0], 0.0));
  if (!(nrm > (double)tau)) return;
  const float scale = (float)((double)tau / nrm);
  TV* vr = v + (size_t)(gl.start[gi] + r0) * d;
  for (long long e = threadIdx.x; e < (long long)n * d; e += blockDim.x)
    vr[e] = from_f<TV>(to_f(vr[e]) * scale);
}

// dst[i] = float(src[i])  (fast-weight reset W <- W_0)
template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ src, float* __restrict__ dst, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = to_f(src[i]);
}

// The fp32 fast weight as two 16-bit planes (tcgen05 path): hi = the upper
// half of the bits rounded half up in magnitude, lo = the signed remainder,
// so that (hi << 16) + lo is the value's bits exactly.
__global__ void split_planes_kernel(const float* __restrict__ w, uint16_t* __restrict__ hi,
                                    uint16_t* __restrict__ lo, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t b = __float_as_uint(w[i]);
    const uint32_t h = (b + 0x8000u) >> 16;
    hi[i] = static_cast<uint16_t>(h);
    lo[i] = static_cast<uint16_t>(b - (h << 16));
  }
}

__global__ void join_planes_kernel(const uint16_t* __restrict__ hi, const uint16_t* __restrict__ lo,
                                   float* __restrict__ w, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    w[i] = __uint_as_float((static_cast<uint32_t>(hi[i]) << 16) +
                           static_cast<uint32_t>(static_cast<int32_t>(static_cast<int16_t>(lo[i]))));
}

// out[c, r] = in[r, c] for an R x Cc matrix (32x32 tiles through shared memory).
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ in, T* __restrict__ out, int R, int Cc) {
  __shared__ T tile[32][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = blockIdx.y * 32 + i;
    if (r < R && c < Cc) tile[i][threadIdx.x] = in[(long long)r * Cc + c];
  }
  __syncthreads();
  const int r2 = blockIdx.y * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c2 = blockIdx.x * 32 + i;
    if (c2 < Cc && r2 < R) out[(long long)c2 * R + r2] = tile[threadIdx.x][i];
  }
}

// x[t] = h[t] / sqrt(mean(h[t]^2) + eps); one block per row.
template <typename TOut>
__global__ void rmsnorm_kernel(const float* __restrict__ h, TOut* __restrict__ x, int d,
                               float eps) {
  const float* hr = h + (long long)blockIdx.x * d;
  float ss = 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(hr[i], hr[i], ss);
  __shared__ float red[32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)d + eps);
  TOut* xr = x + (long long)blockIdx.x * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) xr[i] = from_f<TOut>(hr[i] * inv);
}

// h[t] += o[t], then x[t] = RMSNorm(h[t]) (the next block's input), one block
// per row: the residual add and the next RMSNorm of a pre-norm stack in one
// pass over h.  The same arithmetic in the same order as residual_add_kernel
// followed by rmsnorm_kernel with 256 threads, so the results are identical.
template <typename TO, typename TX>
__global__ void residual_rmsnorm_kernel(float* __restrict__ h, const TO* __restrict__ o,
                                        TX* __restrict__ x, int d, float eps) {
  float* hr = h + (long long)blockIdx.x * d;
  const TO* orow = o + (long long)blockIdx.x * d;
  float ss = 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = hr[i] + to_f(orow[i]);
    hr[i] = v;
    ss = fmaf(v, v, ss);
  }
  __shared__ float red[32];
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0f;
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)d + eps);
  TX* xr = x + (long long)blockIdx.x * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) xr[i] = from_f<TX>(hr[i] * inv);
}

template <typename T>
__global__ void residual_add_kernel(float* __restrict__ h, const T* __restrict__ o, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    h[i] += to_f(o[i]);
}

}  // namespace ttt
