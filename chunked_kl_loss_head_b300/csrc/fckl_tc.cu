// fckl_tc.cu -- the bf16 path on 5th-generation tensor cores (tcgen05) for sm_103a.
//
// One persistent, warp-specialized GEMM engine serves every contraction of the loss:
//   warp 0      TMA producer: streams 64-deep K slabs of A and B into a ring of shared-
//               memory stages (128-byte swizzle), completion tracked by mbarriers;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16 per
//               instruction) into one of two TMEM accumulators and commits each stage
//               back to the producer when the tensor core has read it;
//   warps 2-5   epilogue: tcgen05.ld of the finished accumulator, one tile row per
//               thread, while the MMA warp already fills the other accumulator.
// The epilogue is what makes each GEMM a step of the loss:
//   FwdEpi   logit tile -> running max / sum of exp per row + student logits at the
//            teacher ids (the tile is never written out);
//   BwdEpi   recomputed logit tile -> G = (softmax - p_teacher) * g / (tau N) in bf16;
//   F32Epi   plain fp32 store / accumulate (dW, dH and the engine's test hook).
#include <cuda_bf16.h>

#include <atomic>
#include <cfloat>
#include <climits>
#include <initializer_list>

#include "fckl_internal.h"
#include "fckl_ptx.cuh"

namespace fckl {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;           // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;    // 6 warps
constexpr int kEpiThreads = 128; // warps 2..5
constexpr int kTmemCols = 512;   // two accumulators of up to 256 fp32 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSmemBudget = 220 * 1024;

template <int BN>
struct Shape {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (kSmemBudget / STAGE) > 8 ? 8 : (kSmemBudget / STAGE);
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + STAGES * STAGE + BAR_BYTES;
};

struct Geom {
  int num_m, num_n, num_k;
};

// Shared flag: a role that gave up on a wait tells the others to stop waiting.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              Ctrl* ctrl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > FCKL_WAIT_NS) {
        *abort_flag = 1;
        if (ctrl) set_status(ctrl, FCKL_ERR_TIMEOUT);
        return false;
      }
      __nanosleep(64);
    }
  }
}

__device__ __forceinline__ int lower_bound_ids(const int32_t* ids, int K, int64_t lo) {
  int a = 0, b = K;
  while (a < b) {
    const int m = (a + b) >> 1;
    if (static_cast<int64_t>(ids[m]) < lo) a = m + 1; else b = m;
  }
  return a;
}

__device__ __forceinline__ float pick32(const uint32_t (&v)[32], int j) {
  uint32_t x = v[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) x = (j == i) ? v[i] : x;
  return __uint_as_float(x);
}

// ----------------------------------------------------------------------------------------
// Epilogues.  run() is called by every epilogue thread for every tile; `taddr` addresses
// the thread's TMEM lane (tile row r) at the accumulator's first column.  tcgen05.ld is
// warp-collective, so loops over columns are uniform across the warp and only the
// memory traffic is predicated on the row.

// Forward logit tile (256 vocab columns): per-row (max, sum) of exp2(z * log2e / tau)
// over the tile's columns, and z at every teacher id that falls in the tile.
struct FwdEpi {
  int64_t rows, V;
  float c2;  // log2(e) / tau
  const int32_t* sidx;
  int K;
  float* zk;
  float2* part;
  int nvt;
  Ctrl* ctrl;

  template <int BN>
  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r) const {
    const int64_t row = static_cast<int64_t>(m_t) * BM + r;
    const bool live = row < rows;
    const int64_t n0 = static_cast<int64_t>(n_t) * BN;
    const int32_t* ids = sidx + (live ? row : 0) * K;
    int k = live ? lower_bound_ids(ids, K, n0) : K;
    int64_t nid = (k < K) ? ids[k] : INT64_MAX;
    float m_run = -INFINITY, s_run = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0 + c >= V) break;
      uint32_t v[32];
      tmem_ld_32x32(taddr + c, v);
      tmem_ld_wait();
      float u[32];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        u[i] = (n0 + c + i < V) ? __uint_as_float(v[i]) * c2 : -INFINITY;
        mx = fmaxf(mx, u[i]);
      }
      if (mx > m_run) {
        s_run *= exp2f(m_run - mx);
        m_run = mx;
      }
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) s += exp2f(u[i] - m_run);
      s_run += s;
      while (nid < n0 + c + 32) {
        zk[row * K + k] = pick32(v, static_cast<int>(nid - (n0 + c)));
        ++k;
        nid = (k < K) ? ids[k] : INT64_MAX;
      }
    }
    if (live) part[row * nvt + n_t] = make_float2(m_run, s_run);
  }
};

// Backward logit tile of a vocab stripe [s0, s0 + S): G = (exp(s - lse) - p) * alpha,
// alpha = g / (tau N) for valid rows and 0 for ignored rows, stored as bf16 [rows, ldG].
struct BwdEpi {
  int64_t rows, V, s0, S, ldG;
  float c2;
  const int32_t* sidx;
  const float* sp;
  int K;
  const float* lse;
  const uint8_t* valid;
  Ctrl* ctrl;
  __nv_bfloat16* G;

  template <int BN>
  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r) const {
    const int64_t row = static_cast<int64_t>(m_t) * BM + r;
    const bool live = row < rows;
    const int64_t n0l = static_cast<int64_t>(n_t) * BN;
    const int64_t n0 = s0 + n0l;
    const int64_t vend = (s0 + S < V) ? s0 + S : V;
    float lse2 = 0.f, a = 0.f;
    const int32_t* ids = sidx + (live ? row : 0) * K;
    int k = K;
    if (live) {
      lse2 = lse[row] * kLog2e;
      a = valid[row] ? ctrl->grad_alpha : 0.f;
      k = lower_bound_ids(ids, K, n0);
    }
    int64_t nid = (k < K) ? ids[k] : INT64_MAX;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0l + c >= S) break;
      uint32_t v[32];
      tmem_ld_32x32(taddr + c, v);
      tmem_ld_wait();
      float g[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        g[i] = (n0 + c + i < vend) ? exp2f(__uint_as_float(v[i]) * c2 - lse2) : 0.f;
      while (nid < n0 + c + 32) {
        const int j = static_cast<int>(nid - (n0 + c));
        const float pk = sp[row * K + k];
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] -= (i == j) ? pk : 0.f;
        ++k;
        nid = (k < K) ? ids[k] : INT64_MAX;
      }
      if (live) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * i] * a, g[2 * i + 1] * a);
          w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        uint4* dst = reinterpret_cast<uint4*>(G + row * ldG + n0l + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
    }
  }
};

// fp32 result tile: out[row, col] = acc (+ out when accumulate); with out_bf16 set, the
// (accumulated) value goes to out_bf16 as bf16 instead.  N and ldo are multiples of 4.
struct F32Epi {
  float* out;
  int64_t ldo, M, N;
  int accumulate;
  __nv_bfloat16* out_bf16;
  Ctrl* ctrl;

  template <int BN>
  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r) const {
    const int64_t row = static_cast<int64_t>(m_t) * BM + r;
    const bool live = row < M;
    const int64_t n0 = static_cast<int64_t>(n_t) * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0 + c >= N) break;
      uint32_t v[32];
      tmem_ld_32x32(taddr + c, v);
      tmem_ld_wait();
      if (!live) continue;
      float* o = out + row * ldo + n0 + c;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (n0 + c + 4 * q >= N) break;
        float4 x = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                               __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        if (accumulate) {
          const float4 y = *reinterpret_cast<const float4*>(o + 4 * q);
          x.x += y.x;
          x.y += y.y;
          x.z += y.z;
          x.w += y.w;
        }
        if (out_bf16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
          uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
          *reinterpret_cast<uint2*>(out_bf16 + row * ldo + n0 + c + 4 * q) = pk;
        } else {
          *reinterpret_cast<float4*>(o + 4 * q) = x;
        }
      }
    }
  }
};

// ----------------------------------------------------------------------------------------
// The engine.  A_MN / B_MN select the operand layouts:
//   A K-major: A[m, k] at row m of a [M, K] tensor (TMA box 64 x 128);
//   A MN-major: A[m, k] at row k of a [K, M] tensor (two 64 x 64 boxes per stage);
//   B K-major: B[n, k] at row n of a [N, K] tensor (box 64 x BN), so D = A . B^T;
//   B MN-major: B[k, n] at row k of a [K, N] tensor (BN/64 boxes of 64 x 64).
template <int BN, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Geom g,
                   Epi epi) {
  using S = Shape<BN>;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S::STAGES * S::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S::STAGES * S::B_BYTES);
  uint64_t* empty = full + S::STAGES;
  uint64_t* tfull = empty + S::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = g.num_m * g.num_n;
  Ctrl* ctrl = epi.ctrl;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m_t = tile % g.num_m, n_t = tile / g.num_m;
        for (int kb = 0; kb < g.num_k; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&empty[s], ph ^ 1, abort_flag, ctrl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], S::STAGE);
          uint8_t* a = sA + s * S::A_BYTES;
          uint8_t* b = sB + s * S::B_BYTES;
          if (!A_MN) {
            tma_load_2d(a, &tmA, &full[s], kb * BK, m_t * BM);
          } else {
            tma_load_2d(a, &tmA, &full[s], m_t * BM, kb * BK);
            tma_load_2d(a + 8192, &tmA, &full[s], m_t * BM + 64, kb * BK);
          }
          if (!B_MN) {
            tma_load_2d(b, &tmB, &full[s], kb * BK, n_t * BN);
          } else {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_load_2d(b + h * 8192, &tmB, &full[s], n_t * BN + h * 64, kb * BK);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++lt) {
        const uint32_t acc = lt & 1, use = lt >> 1;
        if (!wait_or_abort(&tempty[acc], (use & 1) ^ 1, abort_flag, ctrl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < g.num_k; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&full[s], ph, abort_flag, ctrl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + s * S::A_BYTES);
          const uint32_t b_base = smem_u32(sB + s * S::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + k * 2048, 8192, 1024) : sdesc_sw128(a_base + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + k * 2048, 8192, 1024) : sdesc_sw128(b_base + k * 32, 16, 1024);
            umma_f16(d_tmem, ad, bd, IDESC, (kb | k) != 0);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
    }
  } else {
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;
    uint32_t lt = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++lt) {
      const int m_t = tile % g.num_m, n_t = tile / g.num_m;
      const uint32_t acc = lt & 1, use = lt >> 1;
      if (!wait_or_abort(&tfull[acc], use & 1, abort_flag, ctrl)) break;
      tc_fence_after();
      epi.template run<BN>(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN, m_t, n_t, r);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    // let copies and MMAs already in flight land before the memory they target goes away
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ----------------------------------------------------------------------------------------
// host side

template <int BN, bool A_MN, bool B_MN, class Epi>
cudaError_t run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int64_t M, int64_t N, int64_t K, const Epi& epi,
                     int num_sms, cudaStream_t st) {
  using S = Shape<BN>;
  auto kern = tc_gemm_kernel<BN, A_MN, B_MN, Epi>;
  static std::atomic<uint64_t> configured{0};  // one bit per device: the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  Geom g;
  g.num_m = static_cast<int>((M + BM - 1) / BM);
  g.num_n = static_cast<int>((N + BN - 1) / BN);
  g.num_k = static_cast<int>((K + BK - 1) / BK);
  const int tiles = g.num_m * g.num_n;
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, kThreads, S::SMEM, st>>>(ta, tb, g, epi);
  return cudaGetLastError();
}

// Operand tensor maps.  K-major: rows of the operand are `outer`, K is `inner`.
bool map_kmajor(CUtensorMap* m, const void* base, int64_t inner_k, int64_t outer, int64_t ld_elems, int box_rows) {
  return encode_tmap_bf16_2d(m, base, inner_k, outer, ld_elems * 2, 64, box_rows);
}
bool map_mnmajor(CUtensorMap* m, const void* base, int64_t inner_mn, int64_t outer_k, int64_t ld_elems) {
  return encode_tmap_bf16_2d(m, base, inner_mn, outer_k, ld_elems * 2, 64, 64);
}

template <bool A_MN, bool B_MN, class Epi>
cudaError_t run_gemm_bn(int bn, const CUtensorMap& ta, const CUtensorMap& tb, int64_t M, int64_t N, int64_t K,
                        const Epi& epi, int num_sms, cudaStream_t st) {
  switch (bn) {
    case 256: return run_gemm<256, A_MN, B_MN>(ta, tb, M, N, K, epi, num_sms, st);
    case 192: return run_gemm<192, A_MN, B_MN>(ta, tb, M, N, K, epi, num_sms, st);
    default: return run_gemm<128, A_MN, B_MN>(ta, tb, M, N, K, epi, num_sms, st);
  }
}

// Tile width over the d columns of dW / dH: the widest of 256 / 192 / 128 that wastes
// the least of the last tile.
int pick_bn(int64_t N) {
  int best = 256;
  double best_eff = 0.0;
  for (int bn : {256, 192, 128}) {
    const int64_t tiles = (N + bn - 1) / bn;
    const double eff = static_cast<double>(N) / static_cast<double>(tiles * bn);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = bn;
    }
  }
  return best;
}

}  // namespace

cudaError_t tc_fwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V, float tau,
                         const int32_t* sidx, int32_t K, float* zk, float2* part, int nvt, Ctrl* ctrl,
                         int num_sms, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!map_kmajor(&ta, Hc, d, rows, d, BM) || !map_kmajor(&tb, W, d, V, d, 256)) return cudaErrorInvalidValue;
  FwdEpi e{rows, V, kLog2e / tau, sidx, K, zk, part, nvt, ctrl};
  return run_gemm<256, false, false>(ta, tb, rows, V, d, e, num_sms, st);
}

cudaError_t tc_bwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V, int64_t s0, int64_t S,
                         float tau, const int32_t* sidx, const float* sp, int32_t K, const float* lse,
                         const uint8_t* valid, Ctrl* ctrl, void* G, int64_t ldG, int num_sms,
                         cudaStream_t st) {
  const int64_t s_eff = (V - s0 < S) ? V - s0 : S;
  CUtensorMap ta, tb;
  const void* Ws = static_cast<const __nv_bfloat16*>(W) + s0 * d;
  if (!map_kmajor(&ta, Hc, d, rows, d, BM) || !map_kmajor(&tb, Ws, d, s_eff, d, 256)) return cudaErrorInvalidValue;
  BwdEpi e{rows, V, s0, S, ldG, kLog2e / tau, sidx, sp, K, lse, valid, ctrl, static_cast<__nv_bfloat16*>(G)};
  return run_gemm<256, false, false>(ta, tb, rows, s_eff, d, e, num_sms, st);
}

cudaError_t tc_dW(const void* G, int64_t ldG, const void* Hc, int64_t rows, int64_t d, int64_t S, float* dW_stripe,
                  int accumulate, Ctrl* ctrl, int num_sms, cudaStream_t st) {
  // D[S, d] = G^T . Hc: A = G^T stored [rows, S] (MN-major), B = Hc stored [rows, d] (MN-major)
  CUtensorMap ta, tb;
  if (!map_mnmajor(&ta, G, S, rows, ldG) || !map_mnmajor(&tb, Hc, d, rows, d)) return cudaErrorInvalidValue;
  F32Epi e{dW_stripe, d, S, d, accumulate, nullptr, ctrl};
  return run_gemm_bn<true, true>(pick_bn(d), ta, tb, S, d, rows, e, num_sms, st);
}

cudaError_t tc_dH(const void* G, int64_t ldG, const void* W_stripe, int64_t rows, int64_t d, int64_t S, float* acc,
                  int accumulate, void* out_bf16, Ctrl* ctrl, int num_sms, cudaStream_t st) {
  // D[rows, d] = G . W_s: A = G stored [rows, S] (K-major), B = W_s stored [S, d] (MN-major)
  CUtensorMap ta, tb;
  if (!map_kmajor(&ta, G, S, rows, ldG, BM) || !map_mnmajor(&tb, W_stripe, d, S, d)) return cudaErrorInvalidValue;
  F32Epi e{acc, d, rows, d, accumulate, static_cast<__nv_bfloat16*>(out_bf16), ctrl};
  return run_gemm_bn<false, true>(pick_bn(d), ta, tb, rows, d, S, e, num_sms, st);
}

cudaError_t tc_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K, int a_mn, int b_mn,
                          int num_sms, cudaStream_t st) {
  CUtensorMap ta, tb;
  bool ok = a_mn ? map_mnmajor(&ta, A, M, K, M) : map_kmajor(&ta, A, K, M, K, BM);
  ok = ok && (b_mn ? map_mnmajor(&tb, B, N, K, N) : map_kmajor(&tb, B, K, N, K, 256));
  if (!ok) return cudaErrorInvalidValue;
  F32Epi e{D, N, M, N, 0, nullptr, nullptr};
  if (!a_mn && !b_mn) return run_gemm<256, false, false>(ta, tb, M, N, K, e, num_sms, st);
  if (!a_mn && b_mn) return run_gemm_bn<false, true>(pick_bn(N), ta, tb, M, N, K, e, num_sms, st);
  if (a_mn && !b_mn) return run_gemm<256, true, false>(ta, tb, M, N, K, e, num_sms, st);
  return run_gemm_bn<true, true>(pick_bn(N), ta, tb, M, N, K, e, num_sms, st);
}

}  // namespace fckl
