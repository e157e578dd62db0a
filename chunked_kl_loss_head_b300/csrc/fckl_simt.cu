// fckl_simt.cu -- the float32 path on CUDA cores (FFMA).  One-pass TF32 tensor-core math
// keeps 10 mantissa bits and cannot hold float32 inputs to a 1e-5 relative loss error, so
// float32 work runs here: a logit-tile kernel for the forward (online max/sum per row and
// the gather at the teacher ids), the same tile recomputed for the backward gradient
// tile G, and a strided GEMM for dW and dH.
#include <cfloat>

#include "fckl_internal.h"

namespace fckl {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int SM_ = 32, SN_ = 256, SK_ = 32;  // logit tile: 32 rows x 256 vocab, k-step 32

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// First position k in the ascending ids of a row with ids[k] >= lo.
__device__ __forceinline__ int lower_bound_ids(const int32_t* ids, int K, int64_t lo) {
  int a = 0, b = K;
  while (a < b) {
    const int m = (a + b) >> 1;
    if (static_cast<int64_t>(ids[m]) < lo) a = m + 1; else b = m;
  }
  return a;
}

// acc[r][j] = sum_k Hc[m0 + 4w + r, k] * W[n0 + lane + 32 j, k] for the warp's 4 rows.
__device__ __forceinline__ void logit_tile(const float* __restrict__ Hc, const float* __restrict__ W, int64_t rows,
                                           int64_t d, int64_t vend, int64_t m0, int64_t n0, float (&acc)[4][8],
                                           float (*As)[SK_ + 1], float (*Bs)[SK_ + 1]) {
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[r][j] = 0.f;
  for (int64_t k0 = 0; k0 < d; k0 += SK_) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i, r = e >> 5, c = e & 31;
      As[r][c] = (m0 + r < rows && k0 + c < d) ? Hc[(m0 + r) * d + k0 + c] : 0.f;
    }
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
      const int e = tid + 256 * i, r = e >> 5, c = e & 31;
      Bs[r][c] = (n0 + r < vend && k0 + c < d) ? W[(n0 + r) * d + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < SK_; ++kk) {
      float a[4], b[8];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[4 * w + r][kk];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = Bs[lane + 32 * j][kk];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(a[r], b[j], acc[r][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float pick8(const float (&v)[8], int j) {
  float x = v[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) x = (j == i) ? v[i] : x;
  return x;
}

__global__ void __launch_bounds__(256) simt_fwd_kernel(const float* __restrict__ Hc, const float* __restrict__ W,
                                                      int64_t rows, int64_t d, int64_t V, float c2,
                                                      const int32_t* __restrict__ sidx, int K, float* __restrict__ zk,
                                                      float2* __restrict__ part, int nvt) {
  __shared__ float As[SM_][SK_ + 1];
  __shared__ float Bs[SN_][SK_ + 1];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * SN_;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SM_;
  float acc[4][8];
  logit_tile(Hc, W, rows, d, V, m0, n0, acc, As, Bs);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t row = m0 + 4 * w + r;
    if (row >= rows) break;
    float u[8];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      u[j] = (n0 + lane + 32 * j < V) ? acc[r][j] * c2 : -INFINITY;
      mx = fmaxf(mx, u[j]);
    }
    mx = warp_max(mx);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += exp2f(u[j] - mx);
    s = warp_sum(s);
    if (lane == 0) part[row * nvt + blockIdx.x] = make_float2(mx, s);
    const int32_t* ids = sidx + row * K;
    for (int k = lower_bound_ids(ids, K, n0); k < K; ++k) {
      const int64_t id = ids[k];
      if (id >= n0 + SN_) break;
      const int col = static_cast<int>(id - n0);
      if (lane == (col & 31)) zk[row * K + k] = pick8(acc[r], col >> 5);
    }
  }
}

template <typename GT>
__global__ void __launch_bounds__(256) simt_bwd_kernel(const float* __restrict__ Hc, const float* __restrict__ W,
                                                      int64_t rows, int64_t d, int64_t V, int64_t s0, int64_t S,
                                                      float c2, const int32_t* __restrict__ sidx,
                                                      const float* __restrict__ sp, int K,
                                                      const float* __restrict__ lse,
                                                      const uint8_t* __restrict__ valid, const Ctrl* ctrl,
                                                      GT* __restrict__ G) {
  __shared__ float As[SM_][SK_ + 1];
  __shared__ float Bs[SN_][SK_ + 1];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nl0 = static_cast<int64_t>(blockIdx.x) * SN_;  // stripe-local column
  const int64_t n0 = s0 + nl0;                                  // vocab id
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SM_;
  const int64_t vend = (s0 + S < V) ? s0 + S : V;
  float acc[4][8];
  logit_tile(Hc, W, rows, d, vend, m0, n0, acc, As, Bs);
  const float alpha = ctrl->grad_alpha;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t row = m0 + 4 * w + r;
    if (row >= rows) break;
    const float lse2 = lse[row] * kLog2e;
    const bool on = valid[row] != 0;
    const float a = on ? alpha : 0.f;
    float g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = (n0 + lane + 32 * j < vend) ? exp2f(acc[r][j] * c2 - lse2) : 0.f;
    const int32_t* ids = sidx + row * K;
    for (int k = lower_bound_ids(ids, K, n0); k < K; ++k) {
      const int64_t id = ids[k];
      if (id >= n0 + SN_ || id >= vend) break;
      const int col = static_cast<int>(id - n0);
      if (lane == (col & 31)) {
        const float pk = sp[row * K + k];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] -= (j == (col >> 5)) ? pk : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t cl = nl0 + lane + 32 * j;
      // an ignored row's G is 0 whatever its teacher data hold (NaN * 0 would be NaN)
      if (cl < S) G[row * S + cl] = static_cast<GT>(on ? g[j] * a : 0.f);
    }
  }
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const float* __restrict__ A, int64_t sam, int64_t sak,
                                                       const float* __restrict__ B, int64_t sbk, int64_t sbn,
                                                       float* __restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                                       int64_t K, int beta) {
  __shared__ float As[16][64 + 1];
  __shared__ float Bs[16][64 + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * 64, n0 = static_cast<int64_t>(blockIdx.x) * 64;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i, kk = e >> 6, x = e & 63;
      As[kk][x] = (m0 + x < M && k0 + kk < K) ? A[(m0 + x) * sam + (k0 + kk) * sak] : 0.f;
      Bs[kk][x] = (n0 + x < N && k0 + kk < K) ? B[(k0 + kk) * sbk + (n0 + x) * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n < N) {
        float* c = C + m * ldc + n;
        *c = beta ? *c + acc[i][j] : acc[i][j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt_fwd_tiles(const float* Hc, const float* W, int64_t rows, int64_t d, int64_t V, float tau,
                                  const int32_t* sidx, int32_t K, float* zk, float2* part, int nvt,
                                  cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(nvt), static_cast<unsigned>((rows + SM_ - 1) / SM_));
  simt_fwd_kernel<<<grid, 256, 0, st>>>(Hc, W, rows, d, V, kLog2e / tau, sidx, K, zk, part, nvt);
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_tiles(const float* Hc, const float* W, int64_t rows, int64_t d, int64_t V, int64_t s0,
                                  int64_t S, float tau, const int32_t* sidx, const float* sp, int32_t K,
                                  const float* lse, const uint8_t* valid, const Ctrl* ctrl, float* G,
                                  cudaStream_t st) {
  const int64_t s_eff = (V - s0 < S) ? V - s0 : S;
  const dim3 grid(static_cast<unsigned>((s_eff + SN_ - 1) / SN_), static_cast<unsigned>((rows + SM_ - 1) / SM_));
  simt_bwd_kernel<float><<<grid, 256, 0, st>>>(Hc, W, rows, d, V, s0, S, kLog2e / tau, sidx, sp, K, lse, valid, ctrl,
                                               G);
  return cudaGetLastError();
}

cudaError_t launch_simt_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk, int64_t sbn,
                             float* C, int64_t ldc, int64_t M, int64_t N, int64_t K, int beta, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>((M + 63) / 64));
  simt_gemm_kernel<<<grid, 256, 0, st>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, N, K, beta);
  return cudaGetLastError();
}

}  // namespace fckl
