// fckl_topk.cu -- teacher top-K extraction: per row of a [T, V] logit matrix, the K largest
// logits and their ids, the preparation step of the offline cache the loss consumes
// (getaibook.com, "Preparing Offline Top-K Logits").
//
// Order: value descending, then id ascending, values compared through order-preserving
// unsigned keys of their float32 bit patterns (sign-magnitude flipped), so every row has
// one exact answer even with ties.
//
// One CTA per row, HBM-bound: the row is streamed once.  A strided sample of the row
// (2048 keys) is radix-selected for a key with r sampled keys above it, r chosen so that
// a few times K row entries are expected above it: the filter threshold; the streaming
// pass appends every entry at or above it to a shared-memory candidate list (a 16-byte
// vector is ruled out by one signed max of its raw bits; a thread whose vector has
// candidates takes one shared atomic for them); the candidates, narrowed to about K, are
// then put in (key, id) order by rank counting (or a bitonic sort for long lists).  When the sample misleads (fewer than K
// candidates, or more than the list holds: heavy ties, tiny or adversarial rows) the row
// takes the exact path: a 4-pass radix select of the K-th largest key, then every entry
// above it plus the entries equal to it in id order.
#include <cuda_bf16.h>

#include <cstdint>

#include "fckl_internal.h"

namespace fckl {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kSample = 2048;  // sampled keys per row, 4 per thread
constexpr int kCap = 4096;     // candidates a row may keep (4 CTAs of 512 threads fit an SM)
constexpr unsigned kFull = 0xffffffffu;

struct TkSmem {
  unsigned long long cand[kCap];  // (key << 32) | (0xffffffff - id): larger = earlier in the order
  uint32_t hist[256];
  uint32_t warp_sum[kTkWarps];
  uint32_t count;
  uint32_t thr;
  uint32_t need;
};

__device__ __forceinline__ uint32_t key_of_bits(uint32_t u) { return (u & 0x80000000u) ? ~u : (u | 0x80000000u); }
__device__ __forceinline__ uint32_t bits_of_key(uint32_t k) { return (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k; }

template <class E>
__device__ __forceinline__ uint32_t bits_at(const E* row, int64_t i);
template <>
__device__ __forceinline__ uint32_t bits_at<uint16_t>(const uint16_t* row, int64_t i) {
  return static_cast<uint32_t>(row[i]) << 16;
}
template <>
__device__ __forceinline__ uint32_t bits_at<uint32_t>(const uint32_t* row, int64_t i) {
  return row[i];
}

__device__ __forceinline__ unsigned long long composite(uint32_t key, int64_t id) {
  return (static_cast<unsigned long long>(key) << 32) | (0xffffffffull - static_cast<unsigned long long>(id));
}

// Bitonic sort of n (a power of two) values in shared memory, descending.
template <class U>
__device__ void bitonic_desc(U* s, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kTkThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const U a = s[i], b = s[ixj];
          const bool desc_block = (i & k) == 0;
          if (desc_block ? (a < b) : (a > b)) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Appends (key, id) when `pred`: one shared atomic per warp.  Every lane of the warp must
// call it (the ballot is warp-wide).
__device__ __forceinline__ void append(TkSmem& sm, bool pred, uint32_t key, int64_t id) {
  const unsigned mask = __ballot_sync(kFull, pred);
  if (!mask) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(&sm.count, static_cast<uint32_t>(__popc(mask)));
  base = __shfl_sync(kFull, base, leader);
  if (pred) {
    const uint32_t pos = base + static_cast<uint32_t>(__popc(mask & ((1u << lane) - 1u)));
    if (pos < static_cast<uint32_t>(kCap)) sm.cand[pos] = composite(key, id);
  }
}

// Calls f(key, id, valid) for every entry of the row, the lanes of each warp together (a
// fixed number of iterations per warp, valid = false past the end), vectorized when the
// row is 16-byte aligned.
template <class E, class F>
__device__ __forceinline__ void for_each_key(const E* row, int64_t V, F&& f) {
  constexpr int kVec = 16 / sizeof(E);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  if (addr % 16 == 0) {
    // kUnroll 16-byte loads per thread in flight before any is used
    constexpr int kUnroll = 4;
    const int64_t nvec = V / kVec;
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const int64_t iters = (nvec + kTkThreads - 1) / kTkThreads;
    for (int64_t it0 = 0; it0 < iters; it0 += kUnroll) {
      uint4 q[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t v = (it0 + u) * kTkThreads + threadIdx.x;
        q[u] = v < nvec ? __ldcs(rv + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (it0 + u >= iters) break;  // the same for the whole CTA
        const int64_t v = (it0 + u) * kTkThreads + threadIdx.x;
        const bool ok = v < nvec;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          uint32_t b;
          if (sizeof(E) == 2) b = (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16);
          else b = w[e];
          f(key_of_bits(b), v * kVec + e, ok);
        }
      }
    }
    const int64_t tail0 = nvec * kVec;
    if (tail0 < V) {  // fewer than kVec entries: one warp-wide round
      const int64_t i = tail0 + threadIdx.x;
      const bool ok = i < V;
      f(ok ? key_of_bits(bits_at(row, i)) : 0u, i, ok);
    }
  } else {
    const int64_t iters = (V + kTkThreads - 1) / kTkThreads;
    for (int64_t it = 0; it < iters; ++it) {
      const int64_t i = it * kTkThreads + threadIdx.x;
      const bool ok = i < V;
      f(ok ? key_of_bits(bits_at(row, i)) : 0u, i, ok);
    }
  }
}

// Warp 0 finds, among the 256 bins of sm.hist, the highest bin b such that the bins from
// 255 down to b hold at least `want` entries; stores b in sm.thr and the count of the bins
// above b in sm.need.  Every thread calls it (two barriers).
__device__ __forceinline__ void top_bin(TkSmem& sm, uint32_t want) {
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane l holds bins 255 - 8l .. 248 - 8l (descending)
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = sm.hist[255 - 8 * lane - i];
      sum += c[i];
    }
    uint32_t incl = sum;  // inclusive scan over lanes (bins from the top)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - sum;
    const unsigned hit = __ballot_sync(kFull, incl >= want);
    const int first = hit ? __ffs(hit) - 1 : 31;
    if (lane == first) {
      uint32_t cum = excl;
      int bin = 248 - 8 * lane;
      for (int i = 0; i < 8; ++i) {
        if (cum + c[i] >= want) {
          bin = 255 - 8 * lane - i;
          break;
        }
        cum += c[i];
      }
      sm.thr = static_cast<uint32_t>(bin);
      sm.need = cum;
    }
  }
  __syncthreads();
}

// The filter threshold from the row's sample (4 keys per thread): the largest key of the
// form p << 16 with at least `want` sampled keys at or above it (a two-pass radix select
// on the top 16 key bits; for bf16 rows, whose keys have 16 significant bits, it is the
// want-th largest sampled key itself).
__device__ __forceinline__ uint32_t sample_threshold(TkSmem& sm, const uint32_t (&sk)[4], uint32_t want) {
  for (int b = threadIdx.x; b < 256; b += kTkThreads) sm.hist[b] = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 4; ++e) atomicAdd(&sm.hist[sk[e] >> 24], 1u);
  top_bin(sm, want);
  const uint32_t hi = sm.thr, above = sm.need;
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += kTkThreads) sm.hist[b] = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if ((sk[e] >> 24) == hi) atomicAdd(&sm.hist[(sk[e] >> 16) & 255u], 1u);
  top_bin(sm, want - above);
  const uint32_t thr = (hi << 24) | (sm.thr << 16);
  __syncthreads();
  return thr;
}

// Bit e set when entry e of the 16-byte vector q passes key >= thr.  When the threshold
// is at or above the key of +0 (the usual case: it sits among the row's largest logits),
// that test is a signed compare of the raw bits against the threshold's value bits:
// negative values and negative NaNs have negative patterns, and positive NaNs sort above
// +inf in both orders.  One signed max over the vector then rules out the vectors with no
// passing entry, nearly all of them.  (A bf16 threshold has zero low 16 bits, so a word's
// high entry can be compared without masking off the low one.)  Below +0 the
// order-preserving keys are compared entry by entry.
template <class E>
__device__ __forceinline__ uint32_t vec_hits(const uint4& q, uint32_t thr) {
  constexpr int kVec = 16 / sizeof(E);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t mask = 0;
  if (thr >= 0x80000000u) {
    const int32_t T = static_cast<int32_t>(thr & 0x7fffffffu);
    int32_t m = max(max(static_cast<int32_t>(q.x), static_cast<int32_t>(q.y)),
                    max(static_cast<int32_t>(q.z), static_cast<int32_t>(q.w)));
    if (sizeof(E) == 2)
      m = max(m, max(max(static_cast<int32_t>(q.x << 16), static_cast<int32_t>(q.y << 16)),
                     max(static_cast<int32_t>(q.z << 16), static_cast<int32_t>(q.w << 16))));
    if (m < T) return 0;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const uint32_t bits = (sizeof(E) == 2 && !(e & 1)) ? (w[e >> 1] << 16) : w[sizeof(E) == 2 ? e >> 1 : e];
      mask |= (static_cast<int32_t>(bits) >= T ? 1u : 0u) << e;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      uint32_t bits;
      if (sizeof(E) == 2) bits = (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16);
      else bits = w[e];
      mask |= (key_of_bits(bits) >= thr ? 1u : 0u) << e;
    }
  }
  return mask;
}

// Appends the entries of vector q flagged in `mask` (ids id0, id0 + 1, ...): one shared
// atomic per thread with hits (at the gpt-oss shape about one vector in 25 has any).
template <class E>
__device__ __forceinline__ void append_vec(TkSmem& sm, const uint4& q, uint32_t mask, int64_t id0) {
  uint32_t base = atomicAdd(&sm.count, static_cast<uint32_t>(__popc(mask)));
  while (mask) {
    const int e = __ffs(mask) - 1;
    mask &= mask - 1;
    const int wi = sizeof(E) == 2 ? e >> 1 : e;  // the 32-bit word holding entry e (selects, no local array)
    const uint32_t word = wi == 0 ? q.x : wi == 1 ? q.y : wi == 2 ? q.z : q.w;
    uint32_t bits;
    if (sizeof(E) == 2) bits = (e & 1) ? (word & 0xffff0000u) : (word << 16);
    else bits = word;
    if (base < static_cast<uint32_t>(kCap)) sm.cand[base] = composite(key_of_bits(bits), id0 + e);
    ++base;
  }
}

// The streaming pass of the fast path: appends every entry whose key is >= thr.  Each
// thread keeps four 16-byte loads in flight, then filters the four vectors (vec_hits) and
// appends the few passing entries (append_vec).  Rows that do not start on a 16-byte
// boundary take the generic per-entry walk.
template <class E>
__device__ __forceinline__ void scan_append(TkSmem& sm, const E* row, int64_t V, uint32_t thr) {
  constexpr int kVec = 16 / sizeof(E);
  constexpr int kUnroll = 4;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  if (addr % 16 != 0) {
    for_each_key(row, V, [&](uint32_t key, int64_t id, bool ok) { append(sm, ok && key >= thr, key, id); });
    return;
  }
  const int64_t nvec = V / kVec;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  const int64_t iters = (nvec + kTkThreads - 1) / kTkThreads;
  for (int64_t it0 = 0; it0 < iters; it0 += kUnroll) {
    uint4 q[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t v = (it0 + u) * kTkThreads + threadIdx.x;
      q[u] = v < nvec ? __ldcs(rv + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (it0 + u >= iters) break;  // the same for the whole CTA
      const int64_t v = (it0 + u) * kTkThreads + threadIdx.x;
      if (v < nvec) {
        const uint32_t mask = vec_hits<E>(q[u], thr);
        if (mask) append_vec<E>(sm, q[u], mask, v * kVec);
      }
    }
  }
  const int64_t tail0 = nvec * kVec;
  if (tail0 < V) {
    const int64_t i = tail0 + threadIdx.x;
    const bool ok = i < V;
    const uint32_t key = ok ? key_of_bits(bits_at(row, i)) : 0u;
    append(sm, ok && key >= thr, key, i);
  }
}

// Exclusive prefix of `flag` over the CTA in thread order: returns this thread's rank and
// the CTA total through `total` (the same for every thread).
__device__ __forceinline__ uint32_t cta_rank(TkSmem& sm, bool flag, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned m = __ballot_sync(kFull, flag);
  if (lane == 0) sm.warp_sum[warp] = static_cast<uint32_t>(__popc(m));
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int w = 0; w < kTkWarps; ++w) {
    const uint32_t c = sm.warp_sum[w];
    before += w < warp ? c : 0;
    all += c;
  }
  __syncthreads();
  *total = all;
  return before + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
}

template <class E>
__global__ void __launch_bounds__(kTkThreads) topk_kernel(const E* __restrict__ logits, int64_t V, int K,
                                                          int32_t* __restrict__ out_idx,
                                                          float* __restrict__ out_val) {
  extern __shared__ __align__(16) uint8_t tk_raw[];
  TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
  const int64_t t = blockIdx.x;
  const E* row = logits + t * V;
  const int tid = threadIdx.x;

  // ---- fast path: threshold from a sample, one streaming pass, sort the candidates
  uint32_t thr = 0;  // V <= kCap: keep every entry
  if (V > kCap) {
    const int64_t stride = V / (kSample / 4);
    uint32_t sk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sk[e] = key_of_bits(bits_at(row, tid * stride + e));
    // about 1.5 K + 8 samples' worth of row entries expected at or above the threshold
    int r = static_cast<int>((3ll * K * kSample + 2 * V - 1) / (2 * V)) + 8;
    if (r > kSample - 1) r = kSample - 1;
    thr = sample_threshold(sm, sk, static_cast<uint32_t>(r) + 1);
  }
  if (tid == 0) sm.count = 0;
  __syncthreads();
  scan_append(sm, row, V, thr);
  __syncthreads();
  uint32_t n = sm.count;
  bool exact = n < static_cast<uint32_t>(K) || n > static_cast<uint32_t>(kCap);

  if (exact) {
    // ---- exact path: radix select of the K-th largest key, 8 bits per pass
    uint32_t prefix = 0, pmask = 0;
    uint32_t need = static_cast<uint32_t>(K);
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += kTkThreads) sm.hist[b] = 0;
      __syncthreads();
      for_each_key(row, V, [&](uint32_t key, int64_t, bool ok) {
        if (ok && (key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
      });
      __syncthreads();
      if (tid == 0) {
        uint32_t cum = 0;
        int bin = 0;
        for (int b = 255; b >= 0; --b) {
          if (cum + sm.hist[b] >= need) {
            bin = b;
            break;
          }
          cum += sm.hist[b];
        }
        sm.need = need - cum;
        sm.thr = prefix | (static_cast<uint32_t>(bin) << shift);
      }
      __syncthreads();
      need = sm.need;
      prefix = sm.thr;
      pmask |= 255u << shift;
    }
    // every entry above the K-th largest key (fewer than K), then `need` entries equal to
    // it, the smallest ids first (the row is walked in id order, one CTA-wide round at a time)
    const uint32_t kth = prefix;
    if (tid == 0) sm.count = 0;
    __syncthreads();
    for_each_key(row, V, [&](uint32_t key, int64_t id, bool ok) { append(sm, ok && key > kth, key, id); });
    __syncthreads();
    const uint32_t above = sm.count;
    uint32_t taken = 0;
    const int64_t rounds = (V + kTkThreads - 1) / kTkThreads;
    for (int64_t it = 0; it < rounds && taken < need; ++it) {
      const int64_t i = it * kTkThreads + tid;
      const bool eq = i < V && key_of_bits(bits_at(row, i)) == kth;
      uint32_t total;
      const uint32_t rank = cta_rank(sm, eq, &total);
      if (eq && taken + rank < need) sm.cand[above + taken + rank] = composite(kth, i);
      taken += total;
    }
    n = static_cast<uint32_t>(K);
    __syncthreads();
  }

  // ---- narrow the candidates to about K before sorting: the 16-bit key prefix of the K-th
  // largest candidate (a two-pass radix select over the list) bounds what can be in the
  // answer; the candidates at or above it move to the upper half of the list and only
  // they are sorted.  (For bf16 rows, whose keys have 16 significant bits, they are the K
  // answers plus any ties with the K-th.)  When they would not fit, the whole list is sorted.
  unsigned long long* srt = sm.cand;
  if (n > static_cast<uint32_t>(K) && n <= static_cast<uint32_t>(kCap / 2)) {
    for (int b = tid; b < 256; b += kTkThreads) sm.hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < static_cast<int>(n); i += kTkThreads)
      atomicAdd(&sm.hist[static_cast<uint32_t>(sm.cand[i] >> 56)], 1u);
    top_bin(sm, static_cast<uint32_t>(K));
    const uint32_t hi = sm.thr, above = sm.need;
    __syncthreads();
    for (int b = tid; b < 256; b += kTkThreads) sm.hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < static_cast<int>(n); i += kTkThreads) {
      const uint32_t key = static_cast<uint32_t>(sm.cand[i] >> 32);
      if ((key >> 24) == hi) atomicAdd(&sm.hist[(key >> 16) & 255u], 1u);
    }
    top_bin(sm, static_cast<uint32_t>(K) - above);
    const uint32_t cut = (hi << 24) | (sm.thr << 16);
    if (tid == 0) sm.count = 0;
    __syncthreads();
    const int rounds = (static_cast<int>(n) + kTkThreads - 1) / kTkThreads;
    for (int r = 0; r < rounds; ++r) {
      const int i = r * kTkThreads + tid;
      const unsigned long long c = i < static_cast<int>(n) ? sm.cand[i] : 0ull;
      const bool keep = i < static_cast<int>(n) && static_cast<uint32_t>(c >> 32) >= cut;
      const unsigned m = __ballot_sync(kFull, keep);
      if (m) {
        const int lane = tid & 31, leader = __ffs(m) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(&sm.count, static_cast<uint32_t>(__popc(m)));
        base = __shfl_sync(kFull, base, leader);
        if (keep) {
          const uint32_t pos = base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
          if (pos < static_cast<uint32_t>(kCap / 2)) sm.cand[kCap / 2 + pos] = c;
        }
      }
    }
    __syncthreads();
    const uint32_t kept = sm.count;
    __syncthreads();
    if (kept >= static_cast<uint32_t>(K) && kept <= static_cast<uint32_t>(kCap / 2)) {
      srt = sm.cand + kCap / 2;
      n = kept;
    }
  }

  // ---- order the candidates and write the first K.  With at most one candidate per
  // thread, each thread counts the candidates ahead of its own (all distinct: the id is
  // part of the composite) and writes it at that rank, with no barrier; longer lists are
  // bitonic-sorted (padded with zeros, which sort last).
  if (n <= static_cast<uint32_t>(kTkThreads)) {
    if (static_cast<uint32_t>(tid) < n) {
      const unsigned long long c = srt[tid];
      uint32_t rank = 0;
#pragma unroll 4
      for (uint32_t j = 0; j < n; ++j) rank += srt[j] > c ? 1u : 0u;
      if (rank < static_cast<uint32_t>(K)) {
        out_idx[t * K + rank] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(c & 0xffffffffull));
        out_val[t * K + rank] = __uint_as_float(bits_of_key(static_cast<uint32_t>(c >> 32)));
      }
    }
    return;
  }
  int np2 = 1;
  while (np2 < static_cast<int>(n)) np2 <<= 1;
  for (int i = static_cast<int>(n) + tid; i < np2; i += kTkThreads) srt[i] = 0ull;
  __syncthreads();
  bitonic_desc(srt, np2);
  for (int k = tid; k < K; k += kTkThreads) {
    const unsigned long long c = srt[k];
    const uint32_t key = static_cast<uint32_t>(c >> 32);
    out_idx[t * K + k] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(c & 0xffffffffull));
    out_val[t * K + k] = __uint_as_float(bits_of_key(key));
  }
}

}  // namespace

size_t topk_smem_bytes() { return sizeof(TkSmem); }

cudaError_t launch_topk(const void* logits, int64_t T, int64_t V, int32_t K, fckl_dtype dtype, int32_t* idx,
                        float* val, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const size_t smem = sizeof(TkSmem);
  cudaError_t e;
  if (dtype == FCKL_BF16) {
    e = cudaFuncSetAttribute(topk_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    topk_kernel<uint16_t><<<static_cast<unsigned>(T), kTkThreads, smem, st>>>(static_cast<const uint16_t*>(logits), V,
                                                                              K, idx, val);
  } else {
    e = cudaFuncSetAttribute(topk_kernel<uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    topk_kernel<uint32_t><<<static_cast<unsigned>(T), kTkThreads, smem, st>>>(static_cast<const uint32_t*>(logits), V,
                                                                              K, idx, val);
  }
  return cudaGetLastError();
}

}  // namespace fckl
