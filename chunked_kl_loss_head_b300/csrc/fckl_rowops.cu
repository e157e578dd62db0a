// fckl_rowops.cu -- the per-row steps of the loss: teacher preparation, the per-row
// combine of vocab-tile partials into lse_t and loss_t, the fixed-order mean over rows,
// the gradient scale g / (tau N) and the final bf16 cast of dH.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>

#include "fckl_internal.h"

namespace fckl {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.6931471805599453f;

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

// Teacher preparation for any K up to FCKL_MAX_K, one warp per row (the teacher's top-K
// cache, getaibook.com, "Preparing Offline Top-K Logits"): p = softmax(topk_logits / tau)
// over the K cached ids, log p alongside, and the (id, p, log p) triples sorted by id so
// the logit-tile epilogues can walk a row's ids in vocabulary order.  Ids outside [0, V) are recorded
// as FCKL_ERR_BAD_INDEX and replaced by INT32_MAX with p = 0, so no later step can use
// them as an address or match them to a column.  zk (the student logits at the ids) is
// cleared for the forward tiles to fill.
__global__ void prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ logits,
                            int64_t rows, int K, int64_t V, float tau, int32_t* __restrict__ sidx,
                            float* __restrict__ sp, float* __restrict__ slogp, float* __restrict__ zk,
                            Ctrl* ctrl) {
  extern __shared__ int32_t sh_ids[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (row >= rows) return;
  int32_t* ids = sh_ids + warp * K;
  const int32_t* irow = idx + row * K;
  const float* lrow = logits + row * K;

  float amax = -INFINITY;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    int32_t id = irow[k];
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      id = INT32_MAX;
    }
    ids[k] = id;
    amax = fmaxf(amax, lrow[k] / tau);
  }
  if (__any_sync(kFull, bad) && lane == 0) set_status(ctrl, FCKL_ERR_BAD_INDEX);
  amax = warp_max(amax);
  float sum = 0.f;
  for (int k = lane; k < K; k += 32) sum += expf(lrow[k] / tau - amax);
  sum = warp_sum(sum);
  const float lse_a = amax + logf(sum);
  __syncwarp();

  for (int k = lane; k < K; k += 32) {
    const int32_t id = ids[k];
    int rank = 0;
    for (int j = 0; j < K; ++j) {
      const int32_t o = ids[j];
      rank += (o < id) | ((o == id) & (j < k));
    }
    const float lp = lrow[k] / tau - lse_a;
    const int64_t o = row * K + rank;
    sidx[o] = id;
    slogp[o] = lp;
    sp[o] = (id == INT32_MAX) ? 0.f : expf(lp);
    zk[o] = 0.f;
  }
}

// The same preparation for K <= 128, with the ids sorted by a bitonic network in registers
// instead of ranked by K compares each.  A row's K (id, k) pairs become keys id * 128 + k
// (so equal ids keep their cached order), padded with all-ones keys that sort last, P keys
// per lane (32 P >= K slots).  Key slot e = P * lane + i holds register i of its lane: the
// network's exchanges across P slots or more are shuffles between lanes, shorter ones are
// swaps between a lane's own registers.  Below V = 2^24 - 1 a key fits 32 bits (bad ids as
// 2^24 - 1, after every valid id); otherwise it is 64 bits wide (bad ids as INT32_MAX).
// The sorted keys then pass through shared memory so that the row's outputs are written
// with consecutive lanes on consecutive ids.
constexpr int kPrepWarps = 4;
constexpr int kSmallK = 128;
constexpr int64_t kKey32MaxV = (int64_t(1) << 24) - 1;  // V below this: 32-bit keys

__device__ __forceinline__ uint32_t shfl_xor_key(uint32_t v, int m) { return __shfl_xor_sync(kFull, v, m); }
__device__ __forceinline__ uint64_t shfl_xor_key(uint64_t v, int m) {
  return __shfl_xor_sync(kFull, static_cast<unsigned long long>(v), m);
}

template <int P, class Key>
__global__ void __launch_bounds__(kPrepWarps * 32) prep_small_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ logits, int64_t rows, int K, int64_t V, float tau,
    int32_t* __restrict__ sidx, float* __restrict__ sp, float* __restrict__ slogp, float* __restrict__ zk,
    Ctrl* ctrl) {
  constexpr int N = 32 * P;
  constexpr bool kWide = sizeof(Key) == 8;
  constexpr uint32_t kBadId = kWide ? uint32_t(INT32_MAX) : uint32_t(kKey32MaxV);
  constexpr int kShift = kWide ? 32 : 7;
  __shared__ float sh_lp[kPrepWarps][N];
  __shared__ Key sh_key[kPrepWarps][N];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kPrepWarps + warp;
  if (row >= rows) return;
  const int32_t* irow = idx + row * K;
  const float* lrow = logits + row * K;

  float a[P];
  Key key[P];
  float amax = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int k = i * 32 + lane;
    a[i] = -INFINITY;
    key[i] = ~Key(0);
    if (k < K) {
      const int32_t id = irow[k];
      uint32_t kid = static_cast<uint32_t>(id);
      if (id < 0 || static_cast<int64_t>(id) >= V) {
        bad = true;
        kid = kBadId;
      }
      a[i] = lrow[k] / tau;
      amax = fmaxf(amax, a[i]);
      key[i] = (static_cast<Key>(kid) << kShift) | static_cast<Key>(k);
    }
  }
  if (__any_sync(kFull, bad) && lane == 0) set_status(ctrl, FCKL_ERR_BAD_INDEX);
  amax = warp_max(amax);
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (i * 32 + lane < K) sum += expf(a[i] - amax);
  sum = warp_sum(sum);
  const float lse_a = amax + logf(sum);
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (i * 32 + lane < K) sh_lp[warp][i * 32 + lane] = a[i] - lse_a;

#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= P) {
#pragma unroll
        for (int i = 0; i < P; ++i) {
          const int e = lane * P + i;
          const Key p = shfl_xor_key(key[i], stride / P);
          const bool keep_min = ((e & stride) == 0) == ((e & size) == 0);
          key[i] = keep_min ? (p < key[i] ? p : key[i]) : (p > key[i] ? p : key[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < P; ++i) {
          if (i & stride) continue;
          const int j = i | stride;
          const Key lo = key[i] < key[j] ? key[i] : key[j];
          const Key hi = key[i] < key[j] ? key[j] : key[i];
          const bool asc = ((lane * P + i) & size) == 0;
          key[i] = asc ? lo : hi;
          key[j] = asc ? hi : lo;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < P; ++i) sh_key[warp][lane * P + i] = key[i];
  __syncwarp();
  for (int e = lane; e < K; e += 32) {
    const Key kk = sh_key[warp][e];
    const uint32_t kid = static_cast<uint32_t>(kk >> kShift);
    const int32_t id = kid == kBadId ? INT32_MAX : static_cast<int32_t>(kid);
    const float lp = sh_lp[warp][static_cast<uint32_t>(kk) & (kWide ? 0xffffffffu : 0x7fu)];
    const int64_t o = row * K + e;
    sidx[o] = id;
    slogp[o] = lp;
    sp[o] = (id == INT32_MAX) ? 0.f : expf(lp);
    zk[o] = 0.f;
  }
}

template <int P>
cudaError_t launch_prep_small(const int32_t* idx, const float* logits, int64_t rows, int32_t K, int64_t V,
                              float tau, ChunkScratch s, Ctrl* ctrl, cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>((rows + kPrepWarps - 1) / kPrepWarps);
  if (V < kKey32MaxV)
    prep_small_kernel<P, uint32_t><<<grid, kPrepWarps * 32, 0, st>>>(idx, logits, rows, K, V, tau, s.sidx, s.sp,
                                                                     s.slogp, s.zk, ctrl);
  else
    prep_small_kernel<P, uint64_t><<<grid, kPrepWarps * 32, 0, st>>>(idx, logits, rows, K, V, tau, s.sidx, s.sp,
                                                                     s.slogp, s.zk, ctrl);
  return cudaGetLastError();
}

// Adds a (max, sum) partial q to a running (m, s) pair of the same base-2 units.
__device__ __forceinline__ void merge_partial(float& m, float& s, float qm, float qs) {
  if (qm > m) {
    s = s * exp2f(m - qm) + qs;  // m = -inf at the start: 0 * 0 + qs
    m = qm;
  } else {
    s += qs * exp2f(qm - m);
  }
}

// One warp per row: merge the (max, sum) partials of every 256-wide vocab tile into the
// row's logsumexp, then loss_t = sum_k p_k (log p_k - s_k + lse_t) with s_k = z_k / tau,
// over the pairs with p_k > 0 (0 log 0 = 0); ignored rows get loss_t = 0.
// Partials are in base-2 units (u = z * log2(e) / tau).  Each lane merges its share of the
// partials in one pass: when the rows start on 16-byte boundaries, two partials per 16-byte
// load and eight loads in flight per batch (the batch's max first, then its exponentials);
// otherwise one at a time.  Then the lanes merge theirs.
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const float2* __restrict__ part, int nvt, const float* __restrict__ zk,
                   const float* __restrict__ sp, const float* __restrict__ slogp, const uint8_t* __restrict__ valid,
                   int64_t rows, int K, float tau, float* __restrict__ lse, float* __restrict__ row_loss) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (row >= rows) return;
  const float2* pr = part + row * nvt;
  const bool ok = valid[row] != 0;
  const int64_t b = row * K;
  // the row's first 32 * kPre (p, log p, z) triples are loaded before the partials, so
  // their latency hides under the merge
  constexpr int kPre = 4;
  float pp[kPre], lq[kPre], zz[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int k = lane + 32 * i;
    pp[i] = lq[i] = zz[i] = 0.f;
    if (ok && k < K) {
      pp[i] = sp[b + k];
      lq[i] = slogp[b + k];
      zz[i] = zk[b + k];
    }
  }
  float m = -INFINITY, s = 0.f;
  if ((nvt & 1) == 0 && (reinterpret_cast<uintptr_t>(part) & 15) == 0) {
    // batches of kBatch 16-byte loads per lane, all issued before any is used; a batch
    // moves the lane's max once, then adds its partials without branches
    const float4* p4 = reinterpret_cast<const float4*>(pr);
    const int n4 = nvt >> 1;
    constexpr int kBatch = 8;
    for (int j0 = lane; j0 < n4; j0 += 32 * kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + 32 * i;
        v[i] = (j < n4) ? p4[j] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      }
      float bm = m;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) bm = fmaxf(bm, fmaxf(v[i].x, v[i].z));
      if (bm == -INFINITY) continue;  // nothing but empty partials so far
      s *= exp2f(m - bm);             // m = -inf at the start: s is 0 and stays 0
      m = bm;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) s += v[i].y * exp2f(v[i].x - m) + v[i].w * exp2f(v[i].z - m);
    }
  } else {
    for (int j = lane; j < nvt; j += 32) {
      const float2 q = pr[j];
      merge_partial(m, s, q.x, q.y);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(kFull, m, o), s2 = __shfl_xor_sync(kFull, s, o);
    const float mm = fmaxf(m, m2);
    s = (mm == -INFINITY) ? 0.f : s * exp2f(m - mm) + s2 * exp2f(m2 - mm);
    m = mm;
  }
  const float l = (m + log2f(s)) * kLn2;
  // a pair outside the support of p (cached logit -inf: log p = -inf) adds 0, not 0 * inf
  float acc = 0.f;
  if (ok) {
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const float t = pp[i] * (lq[i] - zz[i] / tau + l);
      acc += (pp[i] > 0.f) ? t : 0.f;
    }
    for (int k = lane + 32 * kPre; k < K; k += 32) {
      const float pk = sp[b + k];
      const float t = pk * (slogp[b + k] - zk[b + k] / tau + l);
      acc += (pk > 0.f) ? t : 0.f;
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    lse[row] = l;
    row_loss[row] = ok ? acc : 0.f;
  }
}

constexpr int kReduceThreads = 1024;

// Block-wide fixed-order sums (one block): each thread adds a strided slice in fp64, then a
// fixed binary tree.  The result depends only on T, never on the chunk size.
__device__ void block_sum2(double& s, long long& n) {
  __shared__ double sh_s[kReduceThreads];
  __shared__ long long sh_n[kReduceThreads];
  sh_s[threadIdx.x] = s;
  sh_n[threadIdx.x] = n;
  __syncthreads();
  for (int w = kReduceThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      sh_s[threadIdx.x] += sh_s[threadIdx.x + w];
      sh_n[threadIdx.x] += sh_n[threadIdx.x + w];
    }
    __syncthreads();
  }
  s = sh_s[0];
  n = sh_n[0];
}

__global__ void __launch_bounds__(kReduceThreads) loss_reduce_kernel(const float* __restrict__ row_loss,
                                                                    const uint8_t* __restrict__ valid,
                                                                    int64_t T, float* loss, Ctrl* ctrl) {
  double s = 0.0;
  long long n = 0;
  for (int64_t i = threadIdx.x; i < T; i += kReduceThreads) {
    const bool ok = valid[i] != 0;
    s += ok ? static_cast<double>(row_loss[i]) : 0.0;
    n += ok;
  }
  block_sum2(s, n);
  if (threadIdx.x == 0) {
    ctrl->n_valid = n;
    ctrl->loss_sum = s;
    *loss = n > 0 ? static_cast<float>(s / static_cast<double>(n)) : 0.f;
  }
}

__global__ void __launch_bounds__(kReduceThreads) grad_scale_kernel(const uint8_t* __restrict__ valid, int64_t T,
                                                                   float tau, float grad_loss,
                                                                   const float* grad_scale, Ctrl* ctrl) {
  double s = 0.0;
  long long n = 0;
  for (int64_t i = threadIdx.x; i < T; i += kReduceThreads) n += valid[i] != 0;
  block_sum2(s, n);
  if (threadIdx.x == 0) {
    double g = grad_loss;
    if (grad_scale) g *= static_cast<double>(*grad_scale);
    ctrl->n_valid = n;
    ctrl->grad_alpha = n > 0 ? static_cast<float>(g / (static_cast<double>(tau) * static_cast<double>(n))) : 0.f;
  }
}

// Data-parallel partials of the last forward: the fp64 loss sum and N.
__global__ void loss_partials_kernel(const Ctrl* ctrl, double* out) {
  out[0] = ctrl->loss_sum;
  out[1] = static_cast<double>(ctrl->n_valid);
}

// From the partials summed over ranks: the mean loss, and this rank's gradient scale
// N_local / N_total, which turns the backward's g / (tau N_local) into g / (tau N_total).
__global__ void loss_finish_kernel(const double* total, const double* local, float* loss, float* grad_scale) {
  const double n = total[1];
  *loss = n > 0.0 ? static_cast<float>(total[0] / n) : 0.f;
  *grad_scale = n > 0.0 ? static_cast<float>(local[1] / n) : 0.f;
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, __nv_bfloat162* __restrict__ dst, int64_t n4) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = src[i];
    dst[2 * i] = __floats2bfloat162_rn(v.x, v.y);
    dst[2 * i + 1] = __floats2bfloat162_rn(v.z, v.w);
  }
}

// out[c, r] = in[r, c] for a [rows, cols] bf16 matrix: 64 x 64 tiles through shared memory
// (rows 66 elements apart, so both the row-wise writes and the column-wise reads spread
// over the banks), 16-byte global loads and stores wherever a tile row is whole and the
// leading dimension and base allow it, element-wise at the edges.
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ in, int64_t rows, int64_t cols, int64_t ld_in,
                                      uint16_t* __restrict__ out, int64_t ld_out) {
  __shared__ __align__(16) uint16_t tile[64][66];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 64, c0 = static_cast<int64_t>(blockIdx.y) * 64;
  const bool vin = ld_in % 8 == 0 && reinterpret_cast<uintptr_t>(in) % 16 == 0;
  const bool vout = ld_out % 8 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
  for (int i = threadIdx.x; i < 512; i += blockDim.x) {
    const int r = i >> 3, v = i & 7;
    const int64_t gr = r0 + r, gc = c0 + v * 8;
    uint32_t* t = reinterpret_cast<uint32_t*>(&tile[r][v * 8]);
    if (gr < rows && vin && gc + 8 <= cols) {
      const uint4 q = *reinterpret_cast<const uint4*>(in + gr * ld_in + gc);
      t[0] = q.x;
      t[1] = q.y;
      t[2] = q.z;
      t[3] = q.w;
    } else {
      for (int e = 0; e < 8; ++e) tile[r][v * 8 + e] = (gr < rows && gc + e < cols) ? in[gr * ld_in + gc + e] : 0;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 512; i += blockDim.x) {
    const int oc = i >> 3, v = i & 7;  // output row c0 + oc, output columns r0 + 8v .. r0 + 8v + 7
    const int64_t orow = c0 + oc, ocol = r0 + v * 8;
    if (orow >= cols) continue;
    uint32_t w[4];
    for (int e = 0; e < 4; ++e)
      w[e] = static_cast<uint32_t>(tile[v * 8 + 2 * e][oc]) | (static_cast<uint32_t>(tile[v * 8 + 2 * e + 1][oc]) << 16);
    if (vout && ocol + 8 <= rows) {
      *reinterpret_cast<uint4*>(out + orow * ld_out + ocol) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int e = 0; e < 8; ++e)
        if (ocol + e < rows) out[orow * ld_out + ocol + e] = tile[v * 8 + e][oc];
    }
  }
}

}  // namespace

cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out, int64_t ld_out,
                                  cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  // rows (the vocabulary when W is transposed) on grid x, whose limit is 2^31 - 1
  if ((cols + 63) / 64 > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((rows + 63) / 64), static_cast<unsigned>((cols + 63) / 64));
  transpose_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(in), rows, cols, ld_in,
                                              static_cast<uint16_t*>(out), ld_out);
  return cudaGetLastError();
}

cudaError_t launch_prep(const int32_t* idx, const float* logits, int64_t rows, int32_t K, int64_t V,
                        float tau, ChunkScratch s, Ctrl* ctrl, cudaStream_t st) {
  if (K <= 32) return launch_prep_small<1>(idx, logits, rows, K, V, tau, s, ctrl, st);
  if (K <= 64) return launch_prep_small<2>(idx, logits, rows, K, V, tau, s, ctrl, st);
  if (K <= kSmallK) return launch_prep_small<4>(idx, logits, rows, K, V, tau, s, ctrl, st);
  constexpr int warps = 4;
  const unsigned grid = static_cast<unsigned>((rows + warps - 1) / warps);
  prep_kernel<<<grid, warps * 32, warps * K * sizeof(int32_t), st>>>(idx, logits, rows, K, V, tau, s.sidx, s.sp,
                                                                     s.slogp, s.zk, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float2* part, int nvt, const float* zk, const float* sp, const float* slogp,
                           const uint8_t* valid, int64_t rows, int32_t K, float tau, float* lse,
                           float* row_loss, cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps);
  combine_kernel<<<grid, kCombineWarps * 32, 0, st>>>(part, nvt, zk, sp, slogp, valid, rows, K, tau, lse, row_loss);
  return cudaGetLastError();
}

cudaError_t launch_loss_reduce(const float* row_loss, const uint8_t* valid, int64_t T, float* loss, Ctrl* ctrl,
                               cudaStream_t st) {
  loss_reduce_kernel<<<1, kReduceThreads, 0, st>>>(row_loss, valid, T, loss, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_grad_scale(const uint8_t* valid, int64_t T, float tau, float grad_loss, const float* grad_scale,
                              Ctrl* ctrl, cudaStream_t st) {
  grad_scale_kernel<<<1, kReduceThreads, 0, st>>>(valid, T, tau, grad_loss, grad_scale, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_loss_partials(const Ctrl* ctrl, double* out, cudaStream_t st) {
  loss_partials_kernel<<<1, 1, 0, st>>>(ctrl, out);
  return cudaGetLastError();
}

cudaError_t launch_loss_finish(const double* total, const double* local, float* loss, float* grad_scale,
                               cudaStream_t st) {
  loss_finish_kernel<<<1, 1, 0, st>>>(total, local, loss, grad_scale);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t st) {
  const int64_t n4 = n / 4;  // n is a multiple of 4 (d % 8 == 0 for dH; checked for the C-ABI cast)
  const int threads = 256;
  int64_t blocks = (n4 + threads - 1) / threads;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (blocks < 1) blocks = 1;
  f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      reinterpret_cast<const float4*>(src), reinterpret_cast<__nv_bfloat162*>(dst), n4);
  return cudaGetLastError();
}

}  // namespace fckl
