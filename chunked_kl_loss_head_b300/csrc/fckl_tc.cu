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
// The backward of one chunk is a single launch over every vocab stripe: G tiles, dH^T
// tiles and dW tiles of all stripes in one tile sequence, ordered by dependency and
// synchronized through per-stripe completion counters (see BwdChunkEpi).
#include <cuda_bf16.h>

#include <atomic>
#include <cfloat>
#include <climits>

#include "fckl_internal.h"
#include "fckl_ptx.cuh"

namespace fckl {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;            // one 128-byte swizzle row of bf16
constexpr int kBNMax = 256;       // widest tile (N) of any problem
constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiThreads = 128;  // warps 2..5
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kTmemCols = 512;    // two accumulators of up to 256 fp32 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSmemMax = 232448;  // opt-in dynamic shared memory per block
constexpr int kMaxProb = 3;

// Shared-memory plan of one CTA.  CG = CTAs per tile (1, or 2 for a CTA pair, where each
// CTA holds 128 rows of A and half of the tile's B rows).  A pipeline stage holds KSUB
// consecutive 64-deep k-blocks ("sub-blocks", each in the layout of one TMA box), so that
// the per-stage costs (a barrier wait, a commit, the expect-tx) are paid once per KSUB
// k-blocks; fewer, larger stages tolerate less memory latency, so the epilogue type
// chooses.
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

// The tensor maps of a launch: per problem an A and a B operand map and an output map
// (fp32 TMA epilogues).  Passed as one __grid_constant__ kernel parameter, so each map
// lives in parameter space where TMA may read it.
struct Maps {
  CUtensorMap a[kMaxProb], b[kMaxProb], o[kMaxProb];
};

// What the engine hands every epilogue besides its TMEM address: the output tensor map
// of the tile's problem (TMA epilogues) and this CTA's staging shared memory.
struct EpiCtx {
  const CUtensorMap* out;
  uint8_t* staging;
};

// One GEMM problem of a launch: D[M, N] = A . B over K, tiled (128 * CG) x bn x 64.
struct Prob {
  int num_m, num_n, num_k;
  int tiles;       // num_m * num_n
  int a_mn, b_mn;  // operand layouts (see the engine)
  int n_fastest;   // raster: consecutive tiles walk N (1) or M (0)
  int group_m;     // M-fastest raster: tile rows per group (0: all), see raster()
  int bn;          // tile width: a multiple of 32 (of 64 for an MN-major B), at most 256
  int N;           // extent of N; with a K-major B the last tile narrows to what is left
};

// A launch: up to three problems and the dynamic tile counter (a word in the workspace
// that reads `base` when the launch starts), or none for static round-robin scheduling.
// Plain launches run the tiles of problem 0, then of 1, then of 2.  A chunk backward
// (`stripes` > 0) runs, for every vocab stripe s of width S, the G tiles (problem 0), the
// dH^T tiles (1) and the dW tiles (2) of that stripe, in the order
//   G(0), G(1), grad(0), G(2), grad(1), ..., G(ns-1), grad(ns-2), grad(ns-1)
// (grad = the dH^T and dW tiles), G(s) writing gradient buffer s % 3; see BwdChunkEpi.
struct Geom {
  Prob p[kMaxProb];
  int nprob;
  int tiles;
  unsigned int* counter;
  unsigned int base;
  int stripes;          // 0 for a plain launch
  int S;                // stripe width (vocab columns; a multiple of 256)
  int last_cols;        // vocab columns of the last stripe
  unsigned int* done_g; // [stripes]: finished G tiles (each CTA of a pair adds one)
  unsigned int* done_w; // [stripes]: finished dH^T and dW tiles
};

constexpr int kGradBuffers = 3;

// A tile: its problem, vocab stripe (chunk backward), position, depth and the coordinate
// offsets of its operands (k: along K; m / n: along the operand's M / N rows).
struct TileRef {
  int prob, stripe, m_t, n_t, num_k;
  int n0, bn;  // first column of the tile (in its problem / stripe) and its width
  int a_k_off, a_m_off, b_k_off, b_n_off;
  int skip;  // entirely outside the vocabulary (chunk backward's last stripe): no work
};

// The tile's columns: [n_t * bn, +bn), except that with a K-major B operand the last tile
// of N narrows to the columns left, rounded up to 32.  Each MMA instruction costs about
// the same to issue whatever its width, so full-width tiles plus one narrow tile beat a
// narrower width that divides N.
__device__ __forceinline__ void tile_cols(const Prob& q, TileRef& r) {
  r.n0 = r.n_t * q.bn;
  r.bn = q.bn;
  if (!q.b_mn && q.N - r.n0 < q.bn) r.bn = (q.N - r.n0 + 31) & ~31;
}

// Tile t's position.  N fastest: row-major over (m, n).  M fastest: the tile rows are
// taken in groups of group_m (the last group may be smaller), and within a group the tiles
// walk M fastest, then N; so the CTAs working at one time share a few B tiles and at most
// group_m tile rows of A, whatever M is.  (The forward's A is the chunk's hidden states:
// a group of 16 pair tile rows is 4096 rows, 23.6 MB at d = 2880, which stays in L2 while
// the vocabulary streams past it; a 16384-row chunk walked whole would cycle 94 MB.)
__device__ __forceinline__ void raster(const Prob& q, int t, int& m_t, int& n_t) {
  if (q.n_fastest) {
    n_t = t % q.num_n;
    m_t = t / q.num_n;
    return;
  }
  const int gfull = q.group_m > 0 && q.group_m < q.num_m ? q.group_m : q.num_m;
  const int per = gfull * q.num_n;
  const int grp = t / per;
  const int r = t - grp * per;
  const int m0 = grp * gfull;
  const int gm = q.num_m - m0 < gfull ? q.num_m - m0 : gfull;
  m_t = m0 + r % gm;
  n_t = r / gm;
}

template <int CG>
__device__ __forceinline__ TileRef tile_of(const Geom& g, int t) {
  TileRef r{};
  if (!g.stripes) {
    int p = 0;
    while (p + 1 < g.nprob && t >= g.p[p].tiles) t -= g.p[p++].tiles;
    r.prob = p;
    raster(g.p[p], t, r.m_t, r.n_t);
    r.num_k = g.p[p].num_k;
    tile_cols(g.p[p], r);
    return r;
  }
  const int nG = g.p[0].tiles, nR = g.p[1].tiles + g.p[2].tiles, ns = g.stripes;
  int s, local, grad;
  if (t < nG) {
    s = 0, local = t, grad = 0;
  } else {
    const int u = (t - nG) / (nG + nR);
    if (u < ns - 1) {
      const int rr = t - nG - u * (nG + nR);
      grad = rr >= nG;
      s = grad ? u : u + 1;
      local = grad ? rr - nG : rr;
    } else {
      s = ns - 1, grad = 1, local = t - nG - (ns - 1) * (nG + nR);
    }
  }
  const int cols = s == ns - 1 ? g.last_cols : g.S;
  const int buf = s % kGradBuffers;
  r.stripe = s;
  if (!grad) {
    // G[rows, S-stripe] = H_chunk . W_s^T: B rows are vocab rows s*S + n
    r.prob = 0;
    raster(g.p[0], local, r.m_t, r.n_t);
    tile_cols(g.p[0], r);
    r.num_k = g.p[0].num_k;
    r.b_n_off = s * g.S;
    r.skip = r.n_t * g.p[0].bn >= cols;
  } else if (local < g.p[1].tiles) {
    // dH^T[d, rows] += W_s^T . G^T: A = W rows (K) s*S.., B = G buffer columns (K) buf*S..
    r.prob = 1;
    raster(g.p[1], local, r.m_t, r.n_t);
    tile_cols(g.p[1], r);
    r.num_k = (cols + BK - 1) / BK;
    r.a_k_off = s * g.S;
    r.b_k_off = buf * g.S;
  } else {
    // dW[s*S + m, d] (+)= G^T . H_chunk: A = G buffer columns (M) buf*S..
    r.prob = 2;
    raster(g.p[2], local - g.p[1].tiles, r.m_t, r.n_t);
    tile_cols(g.p[2], r);
    r.num_k = g.p[2].num_k;
    r.a_m_off = buf * g.S;
    r.skip = r.m_t * BM * CG >= cols;
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

// Waits until a completion counter written by other CTAs reaches `target` (acquire), with
// the same bound and abort protocol as the mbarrier waits.
__device__ __forceinline__ bool wait_counter(const unsigned int* c, unsigned int target, const AbortFlag& af,
                                             Ctrl* ctrl) {
  if (ld_acquire_gpu(c) >= target) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    __nanosleep(128);
    if (ld_acquire_gpu(c) >= target) return true;
    if ((i & 15) == 15) {
      if (*af.local) return false;
      if (global_ns() - t0 > FCKL_WAIT_NS) {
        af.raise();
        if (ctrl) set_status(ctrl, FCKL_ERR_TIMEOUT);
        return false;
      }
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

// 2^x by the PTX ISA's approximate base-2 exponential, ex2.approx.ftz.f32 (subnormal
// results flush to zero).  Its error, a few units in the last place of fp32, is far below
// what the epilogues keep: the bf16 rounding of G, and sums of exponentials whose loss is
// checked to 2e-3 against the fp64 oracle.  The exponentials are the epilogues' bulk of
// instructions, and the epilogue warps share their sub-partitions with the TMA and MMA
// issuing threads.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float pick32(const uint32_t (&v)[32], int j) {
  uint32_t x = v[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) x = (j == i) ? v[i] : x;
  return __uint_as_float(x);
}

// ----------------------------------------------------------------------------------------
// Epilogues.  run() is called by every epilogue thread for every tile; `taddr` addresses
// the thread's TMEM lane (tile row r) at the accumulator's first column and m_blk is the
// 128-row block of the result that this CTA holds.  tcgen05.ld is warp-collective, so
// loops over columns are uniform across the warp and only the memory traffic is predicated
// on the row.  done() is called once per tile by one epilogue thread after all four
// epilogue warps of the CTA have finished it (only when kSignals); before it, lane 0 of
// each of those warps has called settle() (wait for whatever of the warp's writes the
// signal must cover) and fenced toward the async proxy and at GPU scope.

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
  static constexpr bool kSignals = false;

  __device__ __forceinline__ void run(const TileRef& tr, uint32_t taddr, int m_blk, int r, const EpiCtx&,
                                      uint32_t&) const {
    const int64_t row = static_cast<int64_t>(m_blk) * BM + r;
    const bool live = row < rows;
    const int n_t = tr.n_t;
    const int BN = tr.bn;
    const int64_t n0 = tr.n0;
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
      // the max on the raw logits (c2 > 0 keeps the order), the scale folded into the
      // exponent's multiply-add
      float z[32];
      float mz = -INFINITY;
      if (n0 + c + 32 <= V) {  // a whole chunk of vocabulary columns (all but the last tile's end)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          z[i] = __uint_as_float(v[i]);
          mz = fmaxf(mz, z[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          z[i] = (n0 + c + i < V) ? __uint_as_float(v[i]) : -INFINITY;
          mz = fmaxf(mz, z[i]);
        }
      }
      const float mx = mz * c2;
      if (mx > m_run) {
        s_run *= ex2_fast(m_run - mx);
        m_run = mx;
      }
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) s += ex2_fast(fmaf(z[i], c2, -m_run));
      s_run += s;
      while (nid < n0 + c + 32) {
        zk[row * K + k] = pick32(v, static_cast<int>(nid - (n0 + c)));
        ++k;
        nid = (k < K) ? ids[k] : INT64_MAX;
      }
    }
    if (live) part[row * nvt + n_t] = make_float2(m_run, s_run);
  }

  __device__ __forceinline__ void done(const TileRef&) const {}
};

// Staging shared memory of the TMA epilogues: per epilogue warp two 4 KB buffers, each
// holding a 32-row block of 128-byte rows.
constexpr int kWarpStaging = 2 * 32 * 128;
constexpr int kEpiStaging = 4 * kWarpStaging;

// Backward logit tile of vocab stripe s (columns [s0, s0 + S) with s0 = s * S):
// G = (exp(s - lse) - p) * alpha, alpha = g / (tau N), for valid rows and exactly 0 for
// ignored rows, stored as bf16 into gradient buffer s % 3 (columns [buf * S, buf * S + S) of the
// [rows, ldG] buffer, ldG = 3 * S).  Columns at or past V are written as zeros.
// Each epilogue warp owns 32 rows; per 64-column chunk it converts two 32-column TMEM
// loads to bf16, writes the 32 x 64 block (32 rows of 128 bytes, 128-byte swizzle) into
// one of its two 4 KB staging buffers and one lane TMA-stores it through the output map
// (the gradient buffer, 64 x 32 boxes, rows past the chunk clipped).  Whole 128-byte row
// segments then reach L2 from one bulk copy instead of 16-byte stores from every thread.
struct BwdEpi {
  int64_t rows, V, S, ldG;
  float c2;
  const int32_t* sidx;
  const float* sp;
  int K;
  const float* lse;
  const uint8_t* valid;
  Ctrl* ctrl;

  __device__ __forceinline__ void run(const TileRef& tr, uint32_t taddr, int m_blk, int r, const EpiCtx& cx,
                                      uint32_t& seq) const {
    const int lane = r & 31, quad = r >> 5;
    const int64_t row = static_cast<int64_t>(m_blk) * BM + r;
    const int64_t m0 = static_cast<int64_t>(m_blk) * BM + quad * 32;  // this warp's first row
    const bool live = row < rows;
    const int64_t s0 = static_cast<int64_t>(tr.stripe) * S;
    const int BN = tr.bn;
    const int64_t n0l = tr.n0;
    const int64_t n0 = s0 + n0l;
    const int64_t vend = (s0 + S < V) ? s0 + S : V;
    const int64_t xbuf = (tr.stripe % kGradBuffers) * S + n0l;  // buffer column of the tile
    uint8_t* wbuf = cx.staging + quad * kWarpStaging;
    float lse2 = 0.f, a = 0.f;
    const int32_t* ids = sidx + (live ? row : 0) * K;
    int k = K;
    if (live) {
      if (valid[row]) {
        lse2 = lse[row] * kLog2e;
        a = ctrl->grad_alpha;
        k = lower_bound_ids(ids, K, n0);
      } else {
        // ignored row: every exponential is exactly 0 and no p is read, so its G row is 0
        // whatever its teacher data hold (a NaN there would survive a product with 0)
        lse2 = INFINITY;
      }
    }
    int64_t nid = (k < K) ? ids[k] : INT64_MAX;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      if (n0l + c >= S) break;
      uint8_t* buf = wbuf + (seq & 1) * (32 * 128);
      ++seq;
      if (lane == 0) bulk_wait_read<1>();  // the copy issued two chunks ago has read `buf`
      __syncwarp();
      uint8_t* rowp = buf + lane * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t nc = n0 + c + 32 * h;  // vocab column of this 32-column half
        float g[32];
        if (c + 32 * h < BN) {
          uint32_t v[32];
          tmem_ld_32x32(taddr + c + 32 * h, v);
          tmem_ld_wait();
          if (nc + 32 <= vend) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = ex2_fast(__uint_as_float(v[i]) * c2 - lse2);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = (nc + i < vend) ? ex2_fast(__uint_as_float(v[i]) * c2 - lse2) : 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = 0.f;
        }
        while (nid < nc + 32) {
          const int j = static_cast<int>(nid - nc);
          const float pk = sp[row * K + k];
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] -= (i == j) ? pk : 0.f;
          ++k;
          nid = (k < K) ? ids[k] : INT64_MAX;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(g[2 * i] * a, g[2 * i + 1] * a);
          w[i] = *reinterpret_cast<uint32_t*>(&b2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int piece = 4 * h + q;
          *reinterpret_cast<uint4*>(rowp + ((piece ^ (lane & 7)) << 4)) =
              make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && m0 < rows) {
        tma_store_2d(cx.out, buf, static_cast<int32_t>(xbuf + c), static_cast<int32_t>(m0));
        bulk_commit();
      }
    }
  }

  __device__ __forceinline__ void done(const TileRef&) const {}
};

// fp32 result tile through TMA.  Each epilogue warp owns 32 rows of the tile; per
// 32-column chunk it writes a 32 x 32 fp32 block into one of its two 4 KB staging buffers
// (128-byte swizzle: rows of 128 bytes whose 16-byte pieces are permuted by row % 8, so a
// warp's stores hit distinct banks) and one lane issues a TMA reduce-add into the output
// (accumulate) or a TMA store.  The read-modify-write happens in L2 and the epilogue never
// waits on HBM.  With `transpose`, D[m, n] goes to out[n][m]: the block is written
// transposed into the buffer and stored at (x = m, y = n).  The output map has a 32 x 32
// box and clips everything outside the result; y_stripe shifts the rows of a chunk
// backward's dW tile to its vocab stripe.
struct F32Epi {
  int64_t M, N;  // of D
  int accumulate, transpose;
  int64_t y_stripe;  // rows of the output per vocab stripe (0: no shift)
  Ctrl* ctrl;

  static constexpr int kStaging = kEpiStaging;
  static constexpr int kKSub = 2;
  static constexpr bool kSignals = false;

  __device__ __forceinline__ void run(const TileRef& tr, uint32_t taddr, int m_blk, int r, const EpiCtx& cx,
                                      uint32_t& seq) const {
    const int lane = r & 31, quad = r >> 5;
    uint8_t* wbuf = cx.staging + quad * kWarpStaging;
    const int bn = tr.bn;
    const int64_t n0 = tr.n0;
    const int64_t m0 = static_cast<int64_t>(m_blk) * BM + quad * 32;
    const int64_t y0 = static_cast<int64_t>(tr.stripe) * y_stripe;
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
        const int32_t y = static_cast<int32_t>(transpose ? n0 + c : y0 + m0);
        if (accumulate) tma_reduce_add_2d(cx.out, buf, x, y);
        else tma_store_2d(cx.out, buf, x, y);
        bulk_commit();
      }
    }
  }

  __device__ __forceinline__ void done(const TileRef&) const {}
};

// The backward of one chunk in one launch: problem 0 = G tiles (BwdEpi), 1 = dH^T tiles
// (F32Epi, transposed, reduce-added into the chunk's fp32 dH accumulator, which starts at
// zero), 2 = dW tiles (F32Epi, stored on the first chunk, reduce-added after).  Gradient
// stripes rotate through three buffers.  Two kinds of dependency, both on tiles that come
// earlier in the tile order, so a persistent grid always makes progress:
//   a dH^T or dW tile of stripe s reads G(s): it waits for all G tiles of stripe s;
//   a G tile of stripe s >= 3 overwrites the buffer of stripe s - 3: it waits for all
//   dH^T and dW tiles of stripe s - 3.
// The producers of both CTAs of a pair wait on the counters (acquire, then a proxy fence
// before their TMA reads of G); each CTA adds one to its stripe's counter when its
// epilogue has finished a tile (release).  For a G tile every epilogue warp first waits
// until its TMA stores of the tile have completed (settle), so the count covers them.
struct BwdChunkEpi {
  BwdEpi g;
  F32Epi h, w;
  Ctrl* ctrl;
  unsigned int* done_g;
  unsigned int* done_w;

  static constexpr int kStaging = kEpiStaging;
  static constexpr int kKSub = 2;
  static constexpr bool kSignals = true;

  __device__ __forceinline__ void run(const TileRef& tr, uint32_t taddr, int m_blk, int r, const EpiCtx& cx,
                                      uint32_t& seq) const {
    if (tr.prob == 0) g.run(tr, taddr, m_blk, r, cx, seq);
    else if (tr.prob == 1) h.run(tr, taddr, m_blk, r, cx, seq);
    else w.run(tr, taddr, m_blk, r, cx, seq);
  }

  __device__ __forceinline__ void settle(const TileRef& tr) const {
    if (tr.prob == 0) bulk_wait<0>();
  }

  __device__ __forceinline__ void done(const TileRef& tr) const {
    __threadfence();
    if (tr.prob == 0) {
      fence_proxy_async_global();
      atomicAdd(&done_g[tr.stripe], 1u);
    } else {
      atomicAdd(&done_w[tr.stripe], 1u);
    }
  }
};

// ----------------------------------------------------------------------------------------
// The engine.  Per problem, a_mn / b_mn select the operand layouts:
//   A K-major: A[m, k] at row m of a [M, K] tensor (TMA box 64 x 128);
//   A MN-major: A[m, k] at row k of a [K, M] tensor (two 64 x 64 boxes per sub-block);
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
// work.  Both CTAs' loads signal the leader's `full` barrier; the leader's commits arrive
// on both CTAs' `empty` and `tfull` barriers; the peer's epilogue warps release
// accumulators on the leader's `tempty` barrier.
//
// Tiles are handed out by the (leader's) producer warp: from the global counter when
// there is one (each CTA or pair takes the next tile when it is ready for one, which
// balances tiles of different cost), else round-robin; the tile sequence reaches the MMA
// warp and the epilogue warps of both CTAs through a small shared-memory queue.  Tiles
// marked `skip` never enter the queue: the leader counts them as done for the
// dependency counters and moves on.
constexpr int kQueue = 4;

template <class Epi, int CG>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ Maps maps, const Geom g, const Epi epi) {
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
  uint32_t* epi_count = tmem_slot + 2;  // [2]: epilogue warps through the tiles of each accumulator

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // shared::cluster addresses in the other CTA of the pair (unused when CG == 1)
  auto remote = [&](const void* p, uint32_t r) { return mapa_shared(smem_u32(p), r); };
  const AbortFlag af{abort_local, CG == 2 ? remote(const_cast<int*>(abort_local), rank ^ 1u) : 0u};

  Ctrl* ctrl = epi.ctrl;
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
    epi_count[0] = epi_count[1] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < g.nprob; ++p) {
      tma_prefetch_desc(&maps.a[p]);
      tma_prefetch_desc(&maps.b[p]);
      if (Epi::kStaging) tma_prefetch_desc(&maps.o[p]);
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
      const unsigned int g_target = static_cast<unsigned int>(CG * g.p[0].tiles);
      const unsigned int w_target = static_cast<unsigned int>(CG * (g.p[1].tiles + g.p[2].tiles));
      // The next tile index is fetched one tile ahead, so the counter's round trip overlaps
      // the current tile's loads instead of delaying the next tile's first stage.
      auto fetch = [&]() -> int {
        if (g.counter) return static_cast<int>(atomicAdd(g.counter, 1u) - g.base);
        const int v = next_static;
        next_static += units;
        return v;
      };
      int pre = leader ? fetch() : 0;
      // Stripes whose dependency counters this producer has already seen complete (chunk
      // backward): consecutive tiles of one stripe check once.
      int seen_g = -1, seen_w = -1;
      for (int i = 0;; ++i) {
        const int slot = i % kQueue;
        const uint32_t qph = (i / kQueue) & 1;
        int t;
        TileRef tr{};
        if (leader) {
          if (!wait_or_abort(&qempty[slot], qph ^ 1, af, ctrl)) break;
          for (;;) {
            t = pre;
            if (t >= g.tiles) {
              t = -1;
              break;
            }
            pre = fetch();
            tr = tile_of<CG>(g, t);
            if (!tr.skip) break;
            // nothing to compute: count it for both CTAs of the pair
            atomicAdd(tr.prob == 0 ? &g.done_g[tr.stripe] : &g.done_w[tr.stripe], static_cast<unsigned int>(CG));
          }
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
          if (t >= 0) tr = tile_of<CG>(g, t);
        }
        if (t < 0) break;
        if (g.stripes) {
          // chunk backward: the tile's inputs (G of its stripe) or its output buffer (the
          // stripe three back) must be ready
          bool ok = true;
          if (tr.prob != 0) {
            if (tr.stripe != seen_g) {
              ok = wait_counter(&g.done_g[tr.stripe], g_target, af, ctrl);
              seen_g = tr.stripe;
            }
          } else if (tr.stripe >= kGradBuffers && tr.stripe - kGradBuffers != seen_w) {
            ok = wait_counter(&g.done_w[tr.stripe - kGradBuffers], w_target, af, ctrl);
            seen_w = tr.stripe - kGradBuffers;
          }
          if (!ok) break;
          fence_proxy_async_global();
        }
        const Prob q = g.p[tr.prob];
        const CUtensorMap* ta = &maps.a[tr.prob];
        const CUtensorMap* tb = &maps.b[tr.prob];
        // bytes of one sub-block, both CTAs' boxes
        const uint32_t tx_sub = static_cast<uint32_t>(CG * S::A_SUB + q.bn * BK * 2);
        const int m_row = (tr.m_t * CG + static_cast<int>(rank)) * BM + tr.a_m_off;
        // a CTA pair splits the tile's columns in halves (a narrow last tile too); the box
        // is the problem's full half-width either way, its excess rows unused
        const int n_row = tr.n0 + static_cast<int>(rank) * (tr.bn / CG) + tr.b_n_off;
        const int n_stages = (tr.num_k + S::KSUB - 1) / S::KSUB;
        bool ok = true;
        for (int kb = 0; kb < n_stages; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&empty[s], ph ^ 1, af, ctrl)) {
            ok = false;
            break;
          }
          const int nsub = tr.num_k - kb * S::KSUB < S::KSUB ? tr.num_k - kb * S::KSUB : S::KSUB;
          if (leader) mbar_arrive_expect_tx(&full[s], tx_sub * static_cast<uint32_t>(nsub));
          uint8_t* a = sA + s * S::A_BYTES;
          uint8_t* b = sB + s * S::B_BYTES;
          if (CG == 2) {
            const uint32_t fb = full_leader0 + static_cast<uint32_t>(s) * 8u;
            for (int j = 0; j < nsub; ++j) {
              const int kx = (kb * S::KSUB + j) * BK;
              uint8_t* aj = a + j * S::A_SUB;
              if (!q.a_mn) {
                tma_load_2d_pair(aj, ta, fb, kx + tr.a_k_off, m_row);
              } else {
                tma_load_2d_pair(aj, ta, fb, m_row, kx + tr.a_k_off);
                tma_load_2d_pair(aj + 8192, ta, fb, m_row + 64, kx + tr.a_k_off);
              }
              tma_load_2d_pair(b + j * S::B_SUB, tb, fb, kx + tr.b_k_off, n_row);
            }
          } else {
            const int kx = kb * BK;
            if (!q.a_mn) {
              tma_load_2d(a, ta, &full[s], kx + tr.a_k_off, m_row);
            } else {
              tma_load_2d(a, ta, &full[s], m_row, kx + tr.a_k_off);
              tma_load_2d(a + 8192, ta, &full[s], m_row + 64, kx + tr.a_k_off);
            }
            if (!q.b_mn) {
              tma_load_2d(b, tb, &full[s], kx + tr.b_k_off, n_row);
            } else {
              for (int h = 0; h < q.bn / 64; ++h) tma_load_2d(b + h * 8192, tb, &full[s], n_row + h * 64, kx + tr.b_k_off);
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
        const TileRef tr = tile_of<CG>(g, t);
        const Prob q = g.p[tr.prob];
        const uint32_t idesc = IDESC | (static_cast<uint32_t>(tr.bn >> 3) << 17) |
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
        const int n_stages = (tr.num_k + S::KSUB - 1) / S::KSUB;
        bool ok = true;
        for (int kb = 0; kb < n_stages; ++kb, ++it) {
          const int s = it % S::STAGES;
          const uint32_t ph = (it / S::STAGES) & 1;
          if (!wait_or_abort(&full[s], ph, af, ctrl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = tr.num_k - kb * S::KSUB < S::KSUB ? tr.num_k - kb * S::KSUB : S::KSUB;
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
      const TileRef tr = tile_of<CG>(g, t);
      const uint32_t acc = i & 1, use = i >> 1;
      if (lane == 0) ok = wait_or_abort(&tfull[acc], use & 1, af, ctrl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * kBNMax;
      const int m_blk = tr.m_t * CG + static_cast<int>(rank);  // this CTA's 128-row block
      const EpiCtx cx{&maps.o[tr.prob], staging};
      epi.run(tr, taddr, m_blk, r, cx, seq);
      tc_fence_before();
      if constexpr (Epi::kSignals) {
        // The last of the four epilogue warps through this tile reports it done.  Each warp
        // counts before it releases the accumulator, so no warp can reach the next use of
        // the same counter (two tiles later) before all four have counted this one.  The
        // only wait is settle(): for the warp's own bulk writes of the tile to land.
        __syncwarp();
        if (lane == 0) {
          epi.settle(tr);
          fence_proxy_async_global();
          __threadfence();
          const uint32_t seen = atomicAdd(&epi_count[acc], 1u);
          if (seen == kEpiWarps * use + kEpiWarps - 1) epi.done(tr);
        }
      }
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
  q.group_m = 0;
  q.bn = bn;
  q.N = static_cast<int>(N);
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

// Launches a prepared geometry.  `sched` (may be null) is the dynamic tile counter and the
// host's record of its value, advanced by what this launch consumes (tiles + one final
// fetch per scheduling unit), so the next launch on the stream knows its base without a
// reset.  The grid never exceeds the co-resident units, which the chunk backward's
// dependency waits rely on.
template <int CG, class Epi>
cudaError_t launch_tc(const Maps& maps, Geom g, const Epi& epi, TileSched* sched, int num_sms, cudaStream_t st) {
  using S = Shape<Epi::kStaging, CG, (CG == 2 ? Epi::kKSub : 1)>;
  static_assert(S::SMEM <= kSmemMax && S::STAGES >= 3, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int max_units = 0;
  e = kernel_units<Epi, CG>(dev, num_sms, &max_units);
  if (e != cudaSuccess) return e;
  if (max_units < 1) return cudaErrorInvalidConfiguration;
  if (g.tiles == 0) return cudaSuccess;
  const int units = g.tiles < max_units ? g.tiles : max_units;
  if (sched && sched->counter) {
    g.counter = sched->counter;
    g.base = sched->value;
    sched->value += static_cast<unsigned int>(g.tiles + units);
  }
  auto kern = tc_gemm_kernel<Epi, CG>;
  if (CG == 1) {
    kern<<<units, kThreads, S::SMEM, st>>>(maps, g, epi);
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
  return cudaLaunchKernelEx(&cfg, kern, maps, g, epi);
}

Geom plain_geom(const Prob* probs, int nprob) {
  Geom g{};
  g.nprob = nprob;
  for (int p = 0; p < nprob; ++p) {
    g.p[p] = probs[p];
    g.tiles += probs[p].tiles;
  }
  return g;
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

// Tile width over N.  With a K-major B: 256 (the widest MMA), the last tile narrowing to
// what is left (a multiple of 32: the epilogues work in 32-column chunks, and a CTA pair's
// half of B is then a multiple of 16 rows, whole 8-row swizzle atoms); N below 256 gets
// one tile of N rounded up to 32.  An MN-major B loads 64-column boxes and does not
// narrow: the candidate multiple of 64 with the least padded work, counting a fixed cost
// of 32 columns per tile.
int pick_bn(int64_t N, bool b_mn) {
  if (!b_mn) return N >= 256 ? 256 : static_cast<int>((N + 31) / 32 * 32);
  static const int mn[] = {256, 192, 128, 64};
  int best = mn[0];
  int64_t best_cost = INT64_MAX;
  for (int c : mn) {
    const int64_t cost = (N + c - 1) / c * (c + 32);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

// The loss runs every contraction on CTA pairs; the single-CTA engine serves the test hook
// for operand layouts the pair engine does not take (an MN-major B).
constexpr int kLossCG = 2;
// Rows of the forward's tile-row groups (see raster()).
constexpr int kFwdGroupRows = 4096;

}  // namespace

int tc_grad_buffers() { return kGradBuffers; }

namespace {
// One thread waits, through the engine's own bounded wait, on an mbarrier that nothing
// arrives on: the wait gives up after FCKL_WAIT_NS, records FCKL_ERR_TIMEOUT and raises the
// CTA's abort flag, exactly as a stalled pipeline would.
__global__ void wait_timeout_kernel(Ctrl* ctrl) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  const AbortFlag af{&abort_flag, 0u};
  const bool ok = wait_or_abort(&bar, 0, af, ctrl);
  if (ok || !abort_flag) set_status(ctrl, FCKL_ERR_CUDA);  // the wait must have failed and raised the flag
}
}  // namespace

cudaError_t tc_debug_wait_timeout(Ctrl* ctrl, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(ctrl);
  return cudaGetLastError();
}

cudaError_t tc_fwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V, float tau,
                         const int32_t* sidx, int32_t K, float* zk, float2* part, int nvt, Ctrl* ctrl,
                         TileSched* sched, int num_sms, cudaStream_t st) {
  Maps maps;
  if (!map_kmajor(&maps.a[0], Hc, d, rows, d, BM) || !map_kmajor(&maps.b[0], W, d, V, d, kTileV / kLossCG))
    return cudaErrorInvalidValue;
  FwdEpi e{rows, V, kLog2e / tau, sidx, K, zk, part, nvt, ctrl};
  Prob p = make_prob(rows, V, d, kTileV, false, false, false, kLossCG);
  p.group_m = kFwdGroupRows / (BM * kLossCG);
  return launch_tc<kLossCG>(maps, plain_geom(&p, 1), e, sched, num_sms, st);
}

cudaError_t tc_bwd_chunk(const void* Hc, const void* HcT, int64_t ldT, const void* W, int64_t rows, int64_t d,
                         int64_t V, int64_t S, float tau, const int32_t* sidx, const float* sp, int32_t K,
                         const float* lse, const uint8_t* valid, Ctrl* ctrl, void* G, float* dW, int dW_accumulate,
                         float* dH_acc, unsigned int* done_g, unsigned int* done_w, TileSched* sched, int num_sms,
                         cudaStream_t st) {
  constexpr int cg = kLossCG;
  const int64_t ldG = kGradBuffers * S;
  const int stripes = static_cast<int>((V + S - 1) / S);
  const int bn_h = pick_bn(rows, false), bn_w = pick_bn(d, false);
  Maps maps;
  // problem 0, G[rows, S] = H_chunk . W_s^T:   A = H_chunk [rows, d], B = W [V, d] (K-major)
  // problem 1, dH^T[d, rows] += W_s^T . G^T:   A = W stored [V, d] (MN-major, K = vocab),
  //                                            B = G buffer [rows, ldG] (K-major, K = columns)
  // problem 2, dW[S, d] (+)= G^T . H_chunk:    A = G buffer stored [rows, ldG] (MN-major),
  //                                            B = H_chunk^T [d, ldT] (K-major)
  if (!map_kmajor(&maps.a[0], Hc, d, rows, d, BM) || !map_kmajor(&maps.b[0], W, d, V, d, kTileV / cg) ||
      !map_mnmajor(&maps.a[1], W, d, V, d) || !map_kmajor(&maps.b[1], G, ldG, rows, ldG, bn_h / cg) ||
      !map_mnmajor(&maps.a[2], G, ldG, rows, ldG) || !map_kmajor(&maps.b[2], HcT, rows, d, ldT, bn_w / cg) ||
      !encode_tmap_bf16_2d(&maps.o[0], G, ldG, rows, ldG * 2, 64, 32) ||
      !map_out_f32(&maps.o[1], dH_acc, d, rows, d) || !map_out_f32(&maps.o[2], dW, d, V, d))
    return cudaErrorInvalidValue;
  const Prob p[3] = {make_prob(rows, S, d, kTileV, false, false, false, cg),
                     make_prob(d, rows, S, bn_h, true, false, true, cg),
                     make_prob(S, d, rows, bn_w, true, false, true, cg)};
  Geom g = plain_geom(p, 3);
  g.stripes = stripes;
  g.S = static_cast<int>(S);
  g.last_cols = static_cast<int>(V - (stripes - 1) * S);
  g.tiles = stripes * (p[0].tiles + p[1].tiles + p[2].tiles);
  g.done_g = done_g;
  g.done_w = done_w;
  BwdChunkEpi e;
  e.g = BwdEpi{rows, V, S, ldG, kLog2e / tau, sidx, sp, K, lse, valid, ctrl};
  e.h = F32Epi{d, rows, 1, 1, 0, ctrl};
  e.w = F32Epi{S, d, dW_accumulate, 0, S, ctrl};
  e.ctrl = ctrl;
  e.done_g = done_g;
  e.done_w = done_w;
  return launch_tc<cg>(maps, g, e, sched, num_sms, st);
}

cudaError_t tc_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K, int a_mn, int b_mn,
                          int cta_pair, int num_sms, cudaStream_t st) {
  const int cg = cta_pair ? 2 : 1;
  if (cg == 2 && b_mn) return cudaErrorInvalidValue;
  const int bn = pick_bn(N, b_mn != 0);
  Maps maps;
  bool ok = a_mn ? map_mnmajor(&maps.a[0], A, M, K, M) : map_kmajor(&maps.a[0], A, K, M, K, BM);
  ok = ok && (b_mn ? map_mnmajor(&maps.b[0], B, N, K, N) : map_kmajor(&maps.b[0], B, K, N, K, bn / cg));
  ok = ok && map_out_f32(&maps.o[0], D, N, M, N);
  if (!ok) return cudaErrorInvalidValue;
  F32Epi e{M, N, 0, 0, 0, nullptr};
  const Prob p = make_prob(M, N, K, bn, a_mn, b_mn, true, cg);
  if (cg == 2) return launch_tc<2>(maps, plain_geom(&p, 1), e, nullptr, num_sms, st);
  return launch_tc<1>(maps, plain_geom(&p, 1), e, nullptr, num_sms, st);
}

}  // namespace fckl
