// fckl_tc.cu -- the bf16 path on 5th-generation tensor cores (tcgen05) for sm_103a.
//
// One persistent, warp-specialized GEMM engine serves every contraction of the loss.
// The loss runs it on CTA pairs (cta_group::2, 256-row tiles split over the two SMs of a
// TPC); a single-CTA form (128-row tiles) serves the test hook's other operand layouts.
//   warp 0      TMA producer: hands out tiles and streams 64-deep K slabs of A and B
//               into a ring of shared-memory stages (128-byte swizzle), completion
//               tracked by mbarriers;
//   warp 1      MMA issuer: one thread (of the pair's leader CTA) issues tcgen05.mma
//               (M=128 or 256, N=bn, K=16 per instruction) into one of two TMEM
//               accumulators and commits each stage back to the producers when the
//               tensor core has read it;
//   warps 2-5   epilogue: tcgen05.ld of the finished accumulator, one tile row per
//               thread, while the MMA warp already fills the other accumulator.
// The epilogue is what makes each GEMM a step of the loss:
//   FwdEpi   logit tile -> running max / sum of exp per row + student logits at the
//            teacher ids (the tile is never written out);
//   BwdEpi   recomputed logit tile -> G = (softmax - p_teacher) * g / (tau N) in bf16;
//   F32Epi   fp32 tile -> TMA store or TMA reduce-add (dW, dH and the engine's test hook),
//            optionally transposed.
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
constexpr int BK = 64;            // one 128-byte swizzle row of bf16
constexpr int kBNMax = 256;       // widest tile (N) of any problem
constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiThreads = 128;  // warps 2..5
constexpr int kTmemCols = 512;    // two accumulators of up to 256 fp32 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSmemMax = 232448;  // opt-in dynamic shared memory per block

// Shared-memory plan of one CTA.  CG = CTAs per tile (1, or 2 for a CTA pair, where each
// CTA holds 128 rows of A and half of the tile's B rows).  A pipeline stage holds KSUB
// consecutive 64-deep k-blocks ("sub-blocks", each in the layout of one TMA box), so that
// the per-stage costs (a barrier wait, a commit, the expect-tx) are paid once per KSUB
// k-blocks; fewer, larger stages tolerate less memory latency, which the short launches of
// the backward need, so the epilogue type chooses.
template <int STAGING, int CG, int KSUB_>
struct Shape {
  static constexpr int KSUB = KSUB_;
  static constexpr int A_SUB = BM * BK * 2;
  static constexpr int B_SUB = (kBNMax / CG) * BK * 2;
  static constexpr int A_BYTES = KSUB * A_SUB;
  static constexpr int B_BYTES = KSUB * B_SUB;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int FIT = (kSmemMax - 1024 - BAR_BYTES - STAGING) / STAGE;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + STAGING + BAR_BYTES;
};

// What the engine hands every epilogue besides its TMEM address: the output tensor map
// of the tile's problem (TMA epilogues) and this CTA's staging shared memory.
struct EpiCtx {
  const CUtensorMap* out;
  uint8_t* staging;
};

// One GEMM problem of a launch: D[M, N] = A . B over K, tiled 128 x bn x 64.
struct Prob {
  int num_m, num_n, num_k;
  int tiles;       // num_m * num_n
  int a_mn, b_mn;  // operand layouts (see the engine)
  int n_fastest;   // raster: consecutive tiles walk N (1) or M (0)
  int bn;          // tile width: a multiple of 32 (of 64 for an MN-major B), at most 256
};

// A launch: one or two problems (tiles of the second follow those of the first), and the
// dynamic tile counter (a word in the workspace that reads `base` when the launch starts),
// or none for static round-robin scheduling.
struct Geom {
  Prob p[2];
  int nprob;
  int tiles;
  unsigned int* counter;
  unsigned int base;
};

struct TileRef {
  int prob, m_t, n_t;
};

__device__ __forceinline__ TileRef tile_of(const Geom& g, int t) {
  int p = 0;
  if (g.nprob > 1 && t >= g.p[0].tiles) {
    t -= g.p[0].tiles;
    p = 1;
  }
  const Prob q = p ? g.p[1] : g.p[0];
  TileRef r;
  r.prob = p;
  if (q.n_fastest) {
    r.n_t = t % q.num_n;
    r.m_t = t / q.num_n;
  } else {
    r.m_t = t % q.num_m;
    r.n_t = t / q.num_m;
  }
  return r;
}

// Shared flag: a role that gave up on a wait tells the others to stop waiting (in a CTA
// pair, the peer's flag is raised too).  CLUSTER selects an acquire at cluster scope, for
// phases that the peer CTA completes.
struct AbortFlag {
  volatile int* local;
  uint32_t peer;  // shared::cluster address of the peer's flag, 0 without a peer

  __device__ __forceinline__ void raise() const {
    *local = 1;
    if (peer) st_shared_cluster_u32(peer, 1u);
  }
};

template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const AbortFlag& af, Ctrl* ctrl) {
  auto try_wait = [&] { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (try_wait()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    if (try_wait()) return true;
    if ((i & 63) == 63) {
      if (*af.local) return false;
      if (global_ns() - t0 > FCKL_WAIT_NS) {
        af.raise();
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

  static constexpr int kStaging = 0;
  static constexpr int kKSub = 2;

  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r, int BN, const EpiCtx&,
                                      uint32_t&) const {
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

  static constexpr int kStaging = 0;
  static constexpr int kKSub = 1;

  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r, int BN, const EpiCtx&,
                                      uint32_t&) const {
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

// fp32 result tile through TMA.  Each epilogue warp owns 32 rows of the tile; per
// 32-column chunk it writes a 32 x 32 fp32 block into one of its two 4 KB staging buffers
// (128-byte swizzle: rows of 128 bytes whose 16-byte pieces are permuted by row % 8, so a
// warp's stores hit distinct banks) and one lane issues a TMA reduce-add into the output
// (accumulate) or a TMA store (first pass).  The read-modify-write happens in L2 and the
// epilogue never waits on HBM.  With `transpose`, D[m, n] goes to out[n][m]: the block is
// written transposed into the buffer and stored at (x = m, y = n).  The output map has a
// 32 x 32 box and clips everything outside the M x N result.
struct F32Epi {
  int64_t M, N;  // of D
  int accumulate, transpose;
  Ctrl* ctrl;

  static constexpr int kWarpStaging = 2 * 32 * 32 * 4;
  static constexpr int kStaging = 4 * kWarpStaging;
  static constexpr int kKSub = 2;

  __device__ __forceinline__ void run(uint32_t taddr, int m_t, int n_t, int r, int bn, const EpiCtx& cx,
                                      uint32_t& seq) const {
    const int lane = r & 31, quad = r >> 5;
    uint8_t* wbuf = cx.staging + quad * kWarpStaging;
    const int64_t n0 = static_cast<int64_t>(n_t) * bn;
    const int64_t m0 = static_cast<int64_t>(m_t) * BM + quad * 32;
#pragma unroll 1
    for (int c = 0; c < bn; c += 32) {
      if (n0 + c >= N) break;
      uint8_t* buf = wbuf + (seq & 1) * (32 * 32 * 4);
      ++seq;
      if (lane == 0) bulk_wait_read<1>();  // the copy issued two chunks ago has read `buf`
      __syncwarp();
      uint32_t v[32];
      tmem_ld_32x32(taddr + c, v);
      tmem_ld_wait();
      if (!transpose) {
        uint8_t* rowp = buf + lane * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 x = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          *reinterpret_cast<uint4*>(rowp + ((q ^ (lane & 7)) << 4)) = x;
        }
      } else {
        const int piece = lane >> 2, word = (lane & 3) << 2;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          *reinterpret_cast<uint32_t*>(buf + j * 128 + ((piece ^ (j & 7)) << 4) + word) = v[j];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && m0 < M) {
        const int32_t x = static_cast<int32_t>(transpose ? m0 : n0 + c);
        const int32_t y = static_cast<int32_t>(transpose ? n0 + c : m0);
        if (accumulate) tma_reduce_add_2d(cx.out, buf, x, y);
        else tma_store_2d(cx.out, buf, x, y);
        bulk_commit();
      }
    }
  }
};

// ----------------------------------------------------------------------------------------
// The engine.  Per problem, a_mn / b_mn select the operand layouts:
//   A K-major: A[m, k] at row m of a [M, K] tensor (TMA box 64 x 128);
//   A MN-major: A[m, k] at row k of a [K, M] tensor (two 64 x 64 boxes per stage);
//   B K-major: B[n, k] at row n of a [N, K] tensor (box 64 x bn/CG), so D = A . B^T;
//   B MN-major: B[k, n] at row k of a [K, N] tensor (bn/64 boxes of 64 x 64; CG = 1 only).
// (On this part an MN-major B operand costs 12-25% of MMA throughput and an MN-major A
// nothing, so the loss arranges its contractions to have K-major B operands.)
//
// CG = 2 runs each tile on a CTA pair (a cluster of two CTAs on the two SMs of a TPC):
// the tile is 256 rows x bn, each CTA loads its 128 rows of A and half of the bn rows of
// B, and the leader (rank 0) issues cta_group::2 MMAs that read both CTAs' shared memory
// and write each CTA's 128 accumulator rows into its own TMEM.  Per SM, a 64-deep k-block
// then costs 32 KB of operand traffic instead of 48 KB for the same 128 x 256 x 64 MMA
// work, which is what the L2 -> SM path can sustain.  Both CTAs' loads signal the leader's
// `full` barrier; the leader's commits arrive on both CTAs' `empty` and `tfull` barriers;
// the peer's epilogue warps release accumulators on the leader's `tempty` barrier.
//
// Tiles are handed out by the (leader's) producer warp: from the global counter when
// there is one (each CTA or pair takes the next tile when it is ready for one, which
// balances tiles of different cost), else round-robin; the tile sequence reaches the MMA
// warp and the epilogue warps of both CTAs through a small shared-memory queue.
constexpr int kQueue = 4;
constexpr int kEpiWarps = kEpiThreads / 32;

template <class Epi, int CG>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1, Geom g,
                   Epi e0, Epi e1) {
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per tile");
  using S = Shape<Epi::kStaging, CG, (CG == 2 ? Epi::kKSub : 1)>;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM * CG, 8, false, false) & ~(0x3Fu << 17);  // N set per problem
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S::STAGES * S::A_BYTES;
  uint8_t* staging = sB + S::STAGES * S::B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + Epi::kStaging);
  uint64_t* empty = full + S::STAGES;
  uint64_t* tfull = empty + S::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + kQueue;
  int* tileq = reinterpret_cast<int*>(qempty + kQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tileq + kQueue);
  volatile int* abort_local = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // shared::cluster addresses in the other CTA of the pair (unused when CG == 1)
  auto remote = [&](const void* p, uint32_t r) { return mapa_shared(smem_u32(p), r); };
  const AbortFlag af{abort_local, CG == 2 ? remote(const_cast<int*>(abort_local), rank ^ 1u) : 0u};

  Ctrl* ctrl = e0.ctrl;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CG * kEpiWarps);
    }
    // consumers of a queue slot, one arrival per warp: the leader's MMA warp and the
    // epilogue warps of every CTA, plus the peer's producer
    for (int q = 0; q < kQueue; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 1 + CG * kEpiWarps + (CG - 1));
    }
    *abort_local = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    if (Epi::kStaging) tma_prefetch_desc(&tmO0);
    if (g.nprob > 1) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
      if (Epi::kStaging) tma_prefetch_desc(&tmO1);
    }
  }
  if (warp == 1) {
    if (CG == 2) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      int next_static = unit;
      const uint32_t full_leader0 = CG == 2 ? remote(&full[0], 0) : 0u;
      for (int i = 0;; ++i) {
        const int slot = i % kQueue;
        const uint32_t qph = (i / kQueue) & 1;
        int t;
        if (leader) {
          if (!wait_or_abort(&qempty[slot], qph ^ 1, af, ctrl)) break;
          if (g.counter) {
            t = static_cast<int>(atomicAdd(g.counter, 1u) - g.base);
          } else {
            t = next_static;
            next_static += units;
          }
          if (t >= g.tiles) t = -1;
          tileq[slot] = t;
          mbar_arrive(&qfull[slot]);
          if (CG == 2) {
            st_shared_cluster_u32(remote(&tileq[slot], 1), static_cast<uint32_t>(t));
            mbar_arrive_cluster(remote(&qfull[slot], 1));
          }
        } else {
          if (!wait_or_abort<true>(&qfull[slot], qph, af, ctrl)) break;
          t = tileq[slot];
          mbar_arrive_cluster(remote(&qempty[slot], 0));
        }
        if (t < 0) break;
        const TileRef tr = tile_of(g, t);
        const Prob q = tr.prob ? g.p[1] : g.p[0];
        const CUtensorMap* ta = tr.prob ? &tmA1 : &tmA0;
        const CUtensorMap* tb = tr.prob ? &tmB1 : &tmB0;
        // bytes of one sub-block, both CTAs' boxes
        const uint32_t tx_sub = static_cast<uint32_t>(CG * S::A_SUB + q.bn * BK * 2);
        const int m_row = (tr.m_t * CG + static_cast<int>(rank)) * BM;
        const int b_rows = q.bn / CG;
        const int n_stages = (q.num_k + S::KSUB - 1) / S::KSUB;
        bool ok = true;
        for (int kb = 0; kb < n_stages; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&empty[s], ph ^ 1, af, ctrl)) {
            ok = false;
            break;
          }
          const int nsub = q.num_k - kb * S::KSUB < S::KSUB ? q.num_k - kb * S::KSUB : S::KSUB;
          if (leader) mbar_arrive_expect_tx(&full[s], tx_sub * static_cast<uint32_t>(nsub));
          uint8_t* a = sA + s * S::A_BYTES;
          uint8_t* b = sB + s * S::B_BYTES;
          if (CG == 2) {
            const uint32_t fb = full_leader0 + static_cast<uint32_t>(s) * 8u;
            for (int j = 0; j < nsub; ++j) {
              const int kx = (kb * S::KSUB + j) * BK;
              uint8_t* aj = a + j * S::A_SUB;
              if (!q.a_mn) {
                tma_load_2d_pair(aj, ta, fb, kx, m_row);
              } else {
                tma_load_2d_pair(aj, ta, fb, m_row, kx);
                tma_load_2d_pair(aj + 8192, ta, fb, m_row + 64, kx);
              }
              tma_load_2d_pair(b + j * S::B_SUB, tb, fb, kx, tr.n_t * q.bn + static_cast<int>(rank) * b_rows);
            }
          } else {
            if (!q.a_mn) {
              tma_load_2d(a, ta, &full[s], kb * BK, m_row);
            } else {
              tma_load_2d(a, ta, &full[s], m_row, kb * BK);
              tma_load_2d(a + 8192, ta, &full[s], m_row + 64, kb * BK);
            }
            if (!q.b_mn) {
              tma_load_2d(b, tb, &full[s], kb * BK, tr.n_t * q.bn);
            } else {
              for (int h = 0; h < q.bn / 64; ++h)
                tma_load_2d(b + h * 8192, tb, &full[s], tr.n_t * q.bn + h * 64, kb * BK);
            }
          }
        }
        if (!ok) break;
      }
      // Drain: every stage's last fill has been consumed (the commits that say so have
      // landed on this CTA's barriers) before the CTA may leave.
      for (uint32_t j = 0; j < S::STAGES && j < it; ++j) {
        const uint32_t f = it - 1 - j;
        if (!wait_or_abort(&empty[f % S::STAGES], (f / S::STAGES) & 1, af, ctrl)) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      uint32_t it = 0;
      for (int i = 0;; ++i) {
        const int slot = i % kQueue;
        if (!wait_or_abort(&qfull[slot], (i / kQueue) & 1, af, ctrl)) break;
        const int t = tileq[slot];
        mbar_arrive(&qempty[slot]);
        if (t < 0) break;
        const TileRef tr = tile_of(g, t);
        const Prob q = tr.prob ? g.p[1] : g.p[0];
        const uint32_t idesc = IDESC | (static_cast<uint32_t>(q.bn >> 3) << 17) |
                               (static_cast<uint32_t>(q.a_mn) << 15) | (static_cast<uint32_t>(q.b_mn) << 16);
        const uint32_t acc = i & 1, use = i >> 1;
        if (!wait_or_abort(&tempty[acc], (use & 1) ^ 1, af, ctrl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBNMax;
        // Descriptors of stage 0, sub-block 0; the others differ only in the start address
        // field (address >> 4, which stays below 2^14 for any shared-memory offset), so
        // the issue loop adds offsets instead of rebuilding them: one thread issues every
        // MMA, and its instruction count per MMA shows up in the tensor pipe's duty cycle.
        const uint64_t a_desc0 = q.a_mn ? sdesc_sw128(smem_u32(sA), 8192, 1024) : sdesc_sw128(smem_u32(sA), 16, 1024);
        const uint64_t b_desc0 = q.b_mn ? sdesc_sw128(smem_u32(sB), 8192, 1024) : sdesc_sw128(smem_u32(sB), 16, 1024);
        const uint64_t a_kstep = q.a_mn ? 2048 >> 4 : 32 >> 4, b_kstep = q.b_mn ? 2048 >> 4 : 32 >> 4;
        const int n_stages = (q.num_k + S::KSUB - 1) / S::KSUB;
        bool ok = true;
        for (int kb = 0; kb < n_stages; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&full[s], ph, af, ctrl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = q.num_k - kb * S::KSUB < S::KSUB ? q.num_k - kb * S::KSUB : S::KSUB;
#pragma unroll
          for (int j = 0; j < S::KSUB; ++j) {
            if (j < nsub) {
              const uint64_t ad = a_desc0 + static_cast<uint64_t>((s * S::A_BYTES + j * S::A_SUB) >> 4);
              const uint64_t bd = b_desc0 + static_cast<uint64_t>((s * S::B_BYTES + j * S::B_SUB) >> 4);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                if (CG == 2) umma_f16_pair(d_tmem, ad + k * a_kstep, bd + k * b_kstep, idesc, (kb | j | k) != 0);
                else umma_f16(d_tmem, ad + k * a_kstep, bd + k * b_kstep, idesc, (kb | j | k) != 0);
              }
            }
          }
          if (CG == 2) umma_commit_pair(&empty[s], 0x3);
          else umma_commit(&empty[s]);
        }
        if (!ok) break;
        if (CG == 2) umma_commit_pair(&tfull[acc], 0x3);
        else umma_commit(&tfull[acc]);
      }
    }
  } else {
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;
    uint32_t seq = 0;  // staging-buffer sequence of this warp (TMA epilogues)
    const uint32_t m_off = rank;
    // Lane 0 of each warp waits and reads the queue; the warp follows it (tcgen05.ld is
    // warp-collective, so the lanes must not part ways on a timeout).
    for (int i = 0;; ++i) {
      const int slot = i % kQueue;
      int t = -1;
      int ok = 1;
      if (lane == 0) {
        ok = wait_or_abort<CG == 2>(&qfull[slot], (i / kQueue) & 1, af, ctrl);
        if (ok) {
          t = tileq[slot];
          if (leader) mbar_arrive(&qempty[slot]);
          else mbar_arrive_cluster(remote(&qempty[slot], 0));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!ok || t < 0) break;
      const TileRef tr = tile_of(g, t);
      const uint32_t acc = i & 1, use = i >> 1;
      if (lane == 0) ok = wait_or_abort(&tfull[acc], use & 1, af, ctrl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * kBNMax;
      const int m_blk = tr.m_t * CG + static_cast<int>(m_off);  // this CTA's 128-row block
      if (tr.prob) {
        const EpiCtx cx{&tmO1, staging};
        e1.run(taddr, m_blk, tr.n_t, r, g.p[1].bn, cx, seq);
      } else {
        const EpiCtx cx{&tmO0, staging};
        e0.run(taddr, m_blk, tr.n_t, r, g.p[0].bn, cx, seq);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cluster(remote(&tempty[acc], 0));
      }
    }
    if (Epi::kStaging && lane == 0) bulk_wait<0>();  // this warp's TMA writes have landed
  }

  __syncwarp();
  tc_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (*abort_local) {
    // let copies and MMAs already in flight land before the memory they target goes away
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  if (warp == 1) {
    if (CG == 2) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ----------------------------------------------------------------------------------------
// host side

// M granularity of a tile: 128 rows for one CTA, 256 for a pair.
Prob make_prob(int64_t M, int64_t N, int64_t K, int bn, bool a_mn, bool b_mn, bool n_fastest, int cg) {
  Prob q;
  q.num_m = static_cast<int>((M + BM * cg - 1) / (BM * cg));
  q.num_n = static_cast<int>((N + bn - 1) / bn);
  q.num_k = static_cast<int>((K + BK - 1) / BK);
  q.tiles = q.num_m * q.num_n;
  q.a_mn = a_mn;
  q.b_mn = b_mn;
  q.n_fastest = n_fastest;
  q.bn = bn;
  return q;
}

// Per-device launch facts of one kernel instantiation: the shared-memory attribute is set
// once per device and the number of co-resident units (CTAs, or clusters of two) queried.
struct KernelInfo {
  std::atomic<uint64_t> configured{0};
  int units[64] = {};
};

template <class Epi, int CG>
cudaError_t kernel_units(int dev, int num_sms, int* units) {
  using S = Shape<Epi::kStaging, CG, (CG == 2 ? Epi::kKSub : 1)>;
  static KernelInfo info;
  auto kern = tc_gemm_kernel<Epi, CG>;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(info.configured.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    int n = num_sms;
    if (CG == 2) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = S::SMEM;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg);
      if (e != cudaSuccess) return e;
    }
    info.units[dev & 63] = n;
    info.configured.fetch_or(bit);
  }
  *units = info.units[dev & 63];
  return cudaSuccess;
}

// Launches one or two problems.  `sched` (may be null) is the dynamic tile counter and the
// host's record of its value, advanced by what this launch consumes (tiles + one final
// fetch per scheduling unit), so the next launch on the stream knows its base without a
// reset.  maps: A0, B0, A1, B1, O0, O1 (the second problem's entries repeat the first's
// when absent).  The problems must have been made with the same `CG`.
template <int CG, class Epi>
cudaError_t launch_tc(const CUtensorMap* maps, const Prob* probs, int nprob, const Epi& e0, const Epi& e1,
                      TileSched* sched, int num_sms, cudaStream_t st) {
  using S = Shape<Epi::kStaging, CG, (CG == 2 ? Epi::kKSub : 1)>;
  static_assert(S::SMEM <= kSmemMax && S::STAGES >= 3, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int max_units = 0;
  e = kernel_units<Epi, CG>(dev, num_sms, &max_units);
  if (e != cudaSuccess) return e;
  if (max_units < 1) return cudaErrorInvalidConfiguration;
  Geom g{};
  g.nprob = nprob;
  g.p[0] = probs[0];
  g.p[1] = nprob > 1 ? probs[1] : probs[0];
  g.tiles = probs[0].tiles + (nprob > 1 ? probs[1].tiles : 0);
  if (g.tiles == 0) return cudaSuccess;
  const int units = g.tiles < max_units ? g.tiles : max_units;
  if (sched && sched->counter) {
    g.counter = sched->counter;
    g.base = sched->value;
    sched->value += static_cast<unsigned int>(g.tiles + units);
  }
  auto kern = tc_gemm_kernel<Epi, CG>;
  if (CG == 1) {
    kern<<<units, kThreads, S::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], g, e0, e1);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], g, e0, e1);
}

// Operand tensor maps.  K-major: rows of the operand are `outer`, K is `inner`.
bool map_kmajor(CUtensorMap* m, const void* base, int64_t inner_k, int64_t outer, int64_t ld_elems, int box_rows) {
  return encode_tmap_bf16_2d(m, base, inner_k, outer, ld_elems * 2, 64, box_rows);
}
bool map_mnmajor(CUtensorMap* m, const void* base, int64_t inner_mn, int64_t outer_k, int64_t ld_elems) {
  return encode_tmap_bf16_2d(m, base, inner_mn, outer_k, ld_elems * 2, 64, 64);
}
// fp32 output of the TMA epilogue: [rows, cols] with row stride ld, 32 x 32 boxes.
bool map_out_f32(CUtensorMap* m, const float* base, int64_t cols, int64_t rows, int64_t ld) {
  return encode_tmap_f32_2d(m, base, cols, rows, ld * 4, 32, 32);
}

// Tile width over N: the candidate with the least padded work, counting a fixed cost of 32
// columns per tile for its ramp-up and epilogue.  An MN-major B needs a multiple of 64;
// otherwise multiples of 32 are allowed (the epilogues work in 32-column chunks; a CTA
// pair's half of B is then a multiple of 16 rows, whole 8-row swizzle atoms).
int pick_bn(int64_t N, bool b_mn) {
  static const int mn[] = {256, 192, 128, 64};
  static const int km[] = {256, 224, 192, 160, 128, 96, 64, 32};
  const int* c = b_mn ? mn : km;
  const int n = b_mn ? 4 : 8;
  int best = c[0];
  int64_t best_cost = INT64_MAX;
  for (int i = 0; i < n; ++i) {
    const int64_t cost = (N + c[i] - 1) / c[i] * (c[i] + 32);
    if (cost < best_cost) {
      best_cost = cost;
      best = c[i];
    }
  }
  return best;
}

// The loss runs every contraction on CTA pairs; the single-CTA engine serves the test hook
// for operand layouts the pair engine does not take (an MN-major B).
constexpr int kLossCG = 2;

}  // namespace

cudaError_t tc_fwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V, float tau,
                         const int32_t* sidx, int32_t K, float* zk, float2* part, int nvt, Ctrl* ctrl,
                         TileSched* sched, int num_sms, cudaStream_t st) {
  CUtensorMap maps[6];
  if (!map_kmajor(&maps[0], Hc, d, rows, d, BM) || !map_kmajor(&maps[1], W, d, V, d, kTileV / kLossCG))
    return cudaErrorInvalidValue;
  maps[2] = maps[4] = maps[0];
  maps[3] = maps[5] = maps[1];
  FwdEpi e{rows, V, kLog2e / tau, sidx, K, zk, part, nvt, ctrl};
  const Prob p = make_prob(rows, V, d, kTileV, false, false, false, kLossCG);
  return launch_tc<kLossCG>(maps, &p, 1, e, e, sched, num_sms, st);
}

cudaError_t tc_bwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V, int64_t s0, int64_t S,
                         float tau, const int32_t* sidx, const float* sp, int32_t K, const float* lse,
                         const uint8_t* valid, Ctrl* ctrl, void* G, int64_t ldG, TileSched* sched, int num_sms,
                         cudaStream_t st) {
  const int64_t s_eff = (V - s0 < S) ? V - s0 : S;
  CUtensorMap maps[6];
  const void* Ws = static_cast<const __nv_bfloat16*>(W) + s0 * d;
  if (!map_kmajor(&maps[0], Hc, d, rows, d, BM) || !map_kmajor(&maps[1], Ws, d, s_eff, d, kTileV / kLossCG))
    return cudaErrorInvalidValue;
  maps[2] = maps[4] = maps[0];
  maps[3] = maps[5] = maps[1];
  BwdEpi e{rows, V, s0, S, ldG, kLog2e / tau, sidx, sp, K, lse, valid, ctrl, static_cast<__nv_bfloat16*>(G)};
  const Prob p = make_prob(rows, s_eff, d, kTileV, false, false, false, kLossCG);
  return launch_tc<kLossCG>(maps, &p, 1, e, e, sched, num_sms, st);
}

cudaError_t tc_dW_dH(const void* G, int64_t ldG, const void* HcT, int64_t ldT, const void* W_stripe, int64_t rows,
                     int64_t d, int64_t S, float* dW_stripe, int dW_accumulate, float* dH_acc, int dH_accumulate,
                     Ctrl* ctrl, TileSched* sched, int num_sms, cudaStream_t st) {
  // problem 0, dH^T[d, rows] (+)= W_s^T . G^T: A = W_s stored [S, d] (MN-major), B = G stored
  //            [rows, S] (K-major); the epilogue writes it transposed into dH_acc[rows, d].
  // problem 1, dW[S, d] (+)= G^T . Hc: A = G^T stored [rows, S] (MN-major), B = Hc^T stored
  //            [d, ldT] (K-major).
  // The dH tiles (K = S) are the longer ones and go first.  N fastest: the units in flight
  // share their A block.
  constexpr int cg = kLossCG;
  const int bn_h = pick_bn(rows, false), bn_w = pick_bn(d, false);
  CUtensorMap maps[6];
  if (!map_mnmajor(&maps[0], W_stripe, d, S, d) || !map_kmajor(&maps[1], G, S, rows, ldG, bn_h / cg) ||
      !map_mnmajor(&maps[2], G, S, rows, ldG) || !map_kmajor(&maps[3], HcT, rows, d, ldT, bn_w / cg) ||
      !map_out_f32(&maps[4], dH_acc, d, rows, d) || !map_out_f32(&maps[5], dW_stripe, d, S, d))
    return cudaErrorInvalidValue;
  const Prob p[2] = {make_prob(d, rows, S, bn_h, true, false, true, cg),
                     make_prob(S, d, rows, bn_w, true, false, true, cg)};
  F32Epi eh{d, rows, dH_accumulate, 1, ctrl};
  F32Epi ew{S, d, dW_accumulate, 0, ctrl};
  return launch_tc<cg>(maps, p, 2, eh, ew, sched, num_sms, st);
}

cudaError_t tc_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K, int a_mn, int b_mn,
                          int cta_pair, int num_sms, cudaStream_t st) {
  const int cg = cta_pair ? 2 : 1;
  if (cg == 2 && b_mn) return cudaErrorInvalidValue;
  const int bn = pick_bn(N, b_mn != 0);
  CUtensorMap maps[6];
  bool ok = a_mn ? map_mnmajor(&maps[0], A, M, K, M) : map_kmajor(&maps[0], A, K, M, K, BM);
  ok = ok && (b_mn ? map_mnmajor(&maps[1], B, N, K, N) : map_kmajor(&maps[1], B, K, N, K, bn / cg));
  ok = ok && map_out_f32(&maps[4], D, N, M, N);
  if (!ok) return cudaErrorInvalidValue;
  maps[2] = maps[0];
  maps[3] = maps[1];
  maps[5] = maps[4];
  F32Epi e{M, N, 0, 0, nullptr};
  const Prob p = make_prob(M, N, K, bn, a_mn, b_mn, true, cg);
  if (cg == 2) return launch_tc<2>(maps, &p, 1, e, e, nullptr, num_sms, st);
  return launch_tc<1>(maps, &p, 1, e, e, nullptr, num_sms, st);
}

}  // namespace fckl
