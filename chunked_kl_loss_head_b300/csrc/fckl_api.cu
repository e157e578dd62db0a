// fckl_api.cu -- the C-ABI: argument checks, workspace layout, the chunk loop of the
// forward and the chunk x vocab-stripe loop of the backward, TMA descriptor encoding and
// the optional launch instrumentation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "fckl_internal.h"

namespace fckl {
namespace {

constexpr size_t kAlign = 256;
// Vocab columns of one stripe of the bf16 backward.  It keeps three gradient stripes
// G[block, S] bf16 in flight (one being written, two being read), 96 KiB per row of the
// block: 384 MiB for a block of 4096 rows.  Wider stripes mean fewer passes of the block's
// fp32 dH accumulator (one reduce per stripe, each covering S columns of MMA work); the
// gradient buffers do not stay in the 126 MB L2 next to the rest of a block's working set
// at any width that keeps those passes few.  Measured at the gpt-oss shapes (ABAB on one
// box), 8192 columns took 0.8% less time per step than 4096, and 16384 another 0.9% less
// than 8192; the peak device memory grows by 0.1 and 0.18 GiB.
constexpr int64_t kStripeCols = 16384;
// The f32 path keeps one stripe G[block, S] f32 within this budget.
constexpr size_t kStripeBudgetBytesF32 = size_t(64) << 20;
// Rows of one backward block.  The backward works through a chunk in blocks of at most this
// many rows, which bounds the block's dH accumulator (47 MB at d = 2880) and balances its
// per-stripe reduce against the per-block read-modify-write of dW.  Smaller chunks keep
// their own size (and their smaller workspace).
constexpr int64_t kBwdRowBlock = 4096;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Sizes {
  int64_t T, d, V, K;
  int64_t C;   // rows per chunk: one forward launch, and the per-chunk teacher scratch
  int64_t Cb;  // rows per backward block: min(C, kBwdRowBlock)
  int64_t S, nvt, stripes;
  size_t elem;  // bytes of one H / W / dH element
};

// The stripe width S of the backward for blocks of C rows (a multiple of 256 vocab columns).
int64_t stripe_width(int64_t C, int64_t V, size_t elem) {
  const int64_t vpad = (V + kTileV - 1) / kTileV * kTileV;
  int64_t S = kStripeCols;
  if (elem != 2) S = static_cast<int64_t>(kStripeBudgetBytesF32 / (static_cast<size_t>(C) * 4));
  S = S / kTileV * kTileV;
  if (S < kTileV) S = kTileV;
  if (S > vpad) S = vpad;
  return S;
}

struct Layout {
  size_t ctrl, row_loss, sidx, sp, slogp, zk, part, G, done, dHacc, HcT, total;
  int64_t ldT;
};

Layout layout_of(const Sizes& z) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.ctrl = take(kCtrlBytes);
  L.row_loss = take(sizeof(float) * static_cast<size_t>(z.T));
  const size_t ck = static_cast<size_t>(z.C) * static_cast<size_t>(z.K);
  L.sidx = take(4 * ck);
  L.sp = take(4 * ck);
  L.slogp = take(4 * ck);
  L.zk = take(4 * ck);
  L.part = take(8 * static_cast<size_t>(z.C) * static_cast<size_t>(z.nvt));
  // backward block scratch: sized by the block, not the chunk
  L.G = take(static_cast<size_t>(z.Cb) * static_cast<size_t>(z.S) *
             (z.elem == 2 ? 2 * static_cast<size_t>(tc_grad_buffers()) : 4));
  L.done = take(z.elem == 2 ? 2 * sizeof(unsigned int) * static_cast<size_t>(z.stripes) : 0);
  L.dHacc = take(z.elem == 2 ? 4 * static_cast<size_t>(z.Cb) * static_cast<size_t>(z.d) : 0);
  L.ldT = (z.Cb + 7) / 8 * 8;
  L.HcT = take(z.elem == 2 ? 2 * static_cast<size_t>(z.d) * static_cast<size_t>(L.ldT) : 0);
  L.total = off;
  return L;
}

bool sizes_of(int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, fckl_dtype dt, Sizes* z) {
  if (!valid_sizes(T, d, V, K, chunk, dt)) return false;
  z->T = T;
  z->d = d;
  z->V = V;
  z->K = K;
  z->C = T == 0 ? 1 : (chunk < T ? chunk : T);
  z->Cb = z->C < kBwdRowBlock ? z->C : kBwdRowBlock;
  z->elem = dt == FCKL_BF16 ? 2 : 4;
  z->S = stripe_width(z->Cb, V, z->elem);
  z->stripes = (V + z->S - 1) / z->S;
  z->nvt = (V + kTileV - 1) / kTileV;
  return true;
}

// Checks shared by forward and backward.
fckl_status check_common(const void* H, const void* W, const int32_t* idx, const float* logits,
                         const uint8_t* valid, int64_t T, int64_t d, int64_t V, int32_t K, float tau,
                         int64_t chunk, fckl_dtype dt, void* ws, size_t ws_bytes, Sizes* z) {
  if (!sizes_of(T, d, V, K, chunk, dt, z)) return FCKL_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !std::isfinite(tau)) return FCKL_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !idx || !logits || !valid)) return FCKL_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < layout_of(*z).total) return FCKL_ERR_WORKSPACE;
  if (!aligned(idx, 4) || !aligned(logits, 4)) return FCKL_ERR_UNSUPPORTED;
  if (dt == FCKL_BF16) {
    if (d % 8 != 0 || !aligned(H, 16) || !aligned(W, 16)) return FCKL_ERR_UNSUPPORTED;
  } else {
    if (!aligned(H, 4) || !aligned(W, 4)) return FCKL_ERR_UNSUPPORTED;
  }
  return FCKL_OK;
}

ChunkScratch scratch_of(void* ws, const Layout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  ChunkScratch s;
  s.sidx = reinterpret_cast<int32_t*>(b + L.sidx);
  s.sp = reinterpret_cast<float*>(b + L.sp);
  s.slogp = reinterpret_cast<float*>(b + L.slogp);
  s.zk = reinterpret_cast<float*>(b + L.zk);
  s.part = reinterpret_cast<float2*>(b + L.part);
  s.G = b + L.G;
  s.done = reinterpret_cast<unsigned int*>(b + L.done);
  s.dHacc = reinterpret_cast<float*>(b + L.dHacc);
  s.HcT = b + L.HcT;
  s.ldT = L.ldT;
  return s;
}

// ---- instrumentation ------------------------------------------------------------------

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
struct Pending {
  cudaEvent_t a, b;
};
std::vector<Pending> g_pending[FCKL_K_NUM_CLASSES];
std::vector<cudaEvent_t> g_event_pool;
cudaEvent_t g_open[FCKL_K_NUM_CLASSES];
int64_t g_done_launches[FCKL_K_NUM_CLASSES];
double g_done_ms[FCKL_K_NUM_CLASSES];

cudaEvent_t pool_get() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_sizes(int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, fckl_dtype dt) {
  if (T < 0 || d < 1 || V < 1 || K < 1 || K > FCKL_MAX_K || chunk < 1) return false;
  if (dt != FCKL_F32 && dt != FCKL_BF16) return false;
  return V < (int64_t(1) << 31) && T < (int64_t(1) << 31) && d < (int64_t(1) << 31);
}

fckl_status device_info(int* num_sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FCKL_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FCKL_ERR_CUDA;
  if (major != 10 || minor != 3) return FCKL_ERR_UNSUPPORTED;
  return FCKL_OK;
}

void count_launch(fckl_kernel_class) { g_launches.fetch_add(1, std::memory_order_relaxed); }

void prof_begin(fckl_kernel_class cls, cudaStream_t st) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> g(g_prof_mu);
  cudaEvent_t e = pool_get();
  if (e && cudaEventRecord(e, st) == cudaSuccess) g_open[cls] = e;
}

void prof_end(fckl_kernel_class cls, cudaStream_t st) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (!g_open[cls]) return;
  cudaEvent_t e = pool_get();
  if (e && cudaEventRecord(e, st) == cudaSuccess) g_pending[cls].push_back({g_open[cls], e});
  g_open[cls] = nullptr;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

static bool encode_2d(CUtensorMapDataType dt, CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  std::memset(map, 0, sizeof(*map));
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, inner, outer, row_stride_bytes, box_inner, box_outer);
}

bool encode_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_2d(CU_TENSOR_MAP_DATA_TYPE_FLOAT32, map, base, inner, outer, row_stride_bytes, box_inner, box_outer);
}

}  // namespace fckl

using namespace fckl;

extern "C" {

size_t fckl_workspace_size(int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, fckl_dtype dtype) {
  Sizes z;
  if (!sizes_of(T, d, V, K, chunk, dtype, &z)) return 0;
  return layout_of(z).total;
}

fckl_status fckl_forward(const void* H, const void* W, const int32_t* topk_idx, const float* topk_logits,
                         const uint8_t* valid, int64_t T, int64_t d, int64_t V, int32_t K, float tau, int64_t chunk,
                         fckl_dtype dtype, float* loss, float* lse, float* row_loss, void* ws, size_t ws_bytes,
                         void* stream) {
  Sizes z;
  FCKL_TRY(check_common(H, W, topk_idx, topk_logits, valid, T, d, V, K, tau, chunk, dtype, ws, ws_bytes, &z));
  if (!loss || (T > 0 && !lse)) return FCKL_ERR_INVALID_ARG;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout_of(z);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(wsb + L.ctrl);
  float* rl = row_loss ? row_loss : reinterpret_cast<float*>(wsb + L.row_loss);
  ChunkScratch s = scratch_of(ws, L);

  FCKL_TRY(step(FCKL_K_OTHER, st, [&] { return cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st); }));
  TileSched sched{&ctrl->tile_counter, 0};
  const int nvt = static_cast<int>(z.nvt);
  for (int64_t c0 = 0; c0 < T; c0 += z.C) {
    const int64_t rows = (T - c0 < z.C) ? T - c0 : z.C;
    FCKL_TRY(step(FCKL_K_PREP, st, [&] {
      return launch_prep(topk_idx + c0 * K, topk_logits + c0 * K, rows, K, V, tau, s, ctrl, st);
    }));
    if (dtype == FCKL_BF16) {
      const void* Hc = static_cast<const uint8_t*>(H) + c0 * d * 2;
      FCKL_TRY(step(FCKL_K_FWD_TILES, st, [&] {
        return tc_fwd_tiles(Hc, W, rows, d, V, tau, s.sidx, K, s.zk, s.part, nvt, ctrl, &sched, num_sms, st);
      }));
    } else {
      const float* Hc = static_cast<const float*>(H) + c0 * d;
      FCKL_TRY(step(FCKL_K_FWD_TILES, st, [&] {
        return launch_simt_fwd_tiles(Hc, static_cast<const float*>(W), rows, d, V, tau, s.sidx, K, s.zk, s.part, nvt,
                                     st);
      }));
    }
    FCKL_TRY(step(FCKL_K_COMBINE, st, [&] {
      return launch_combine(s.part, nvt, s.zk, s.sp, s.slogp, valid + c0, rows, K, tau, lse + c0, rl + c0, st);
    }));
  }
  FCKL_TRY(step(FCKL_K_REDUCE, st, [&] { return launch_loss_reduce(rl, valid, T, loss, ctrl, st); }));
  return FCKL_OK;
}

fckl_status fckl_backward(const void* H, const void* W, const int32_t* topk_idx, const float* topk_logits,
                          const uint8_t* valid, int64_t T, int64_t d, int64_t V, int32_t K, float tau, int64_t chunk,
                          fckl_dtype dtype, const float* lse, float grad_loss, const float* grad_scale, void* dH,
                          float* dW, void* ws, size_t ws_bytes, void* stream) {
  Sizes z;
  FCKL_TRY(check_common(H, W, topk_idx, topk_logits, valid, T, d, V, K, tau, chunk, dtype, ws, ws_bytes, &z));
  if (!dW || (T > 0 && (!lse || !dH))) return FCKL_ERR_INVALID_ARG;
  if (!std::isfinite(grad_loss)) return FCKL_ERR_INVALID_ARG;
  if (dtype == FCKL_BF16 ? !aligned(dH, 16) : !aligned(dH, 4)) return FCKL_ERR_UNSUPPORTED;
  if (!aligned(dW, 16)) return FCKL_ERR_UNSUPPORTED;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout_of(z);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(wsb + L.ctrl);
  ChunkScratch s = scratch_of(ws, L);

  if (T == 0) {
    return step(FCKL_K_OTHER, st, [&] { return cudaMemsetAsync(dW, 0, sizeof(float) * V * d, st); });
  }
  FCKL_TRY(step(FCKL_K_OTHER, st,
                [&] { return cudaMemsetAsync(&ctrl->tile_counter, 0, sizeof(ctrl->tile_counter), st); }));
  TileSched sched{&ctrl->tile_counter, 0};
  FCKL_TRY(step(FCKL_K_REDUCE, st, [&] { return launch_grad_scale(valid, T, tau, grad_loss, grad_scale, ctrl, st); }));
  const int64_t S = z.S;
  for (int64_t c0 = 0; c0 < T; c0 += z.Cb) {
    const int64_t rows = (T - c0 < z.Cb) ? T - c0 : z.Cb;
    FCKL_TRY(step(FCKL_K_PREP, st, [&] {
      return launch_prep(topk_idx + c0 * K, topk_logits + c0 * K, rows, K, V, tau, s, ctrl, st);
    }));
    if (dtype == FCKL_BF16) {
      // one launch for every stripe of the chunk (recomputed logits -> G -> dH, dW)
      const void* Hc = static_cast<const uint8_t*>(H) + c0 * d * 2;
      FCKL_TRY(step(FCKL_K_OTHER, st, [&] { return launch_transpose_bf16(Hc, rows, d, d, s.HcT, s.ldT, st); }));
      FCKL_TRY(step(FCKL_K_OTHER, st,
                    [&] { return cudaMemsetAsync(s.dHacc, 0, sizeof(float) * static_cast<size_t>(rows * d), st); }));
      FCKL_TRY(step(FCKL_K_OTHER, st, [&] {
        return cudaMemsetAsync(s.done, 0, 2 * sizeof(unsigned int) * static_cast<size_t>(z.stripes), st);
      }));
      FCKL_TRY(step(FCKL_K_BWD_TILES, st, [&] {
        return tc_bwd_chunk(Hc, s.HcT, s.ldT, W, rows, d, V, S, tau, s.sidx, s.sp, K, lse + c0, valid + c0, ctrl,
                            s.G, dW, c0 > 0, s.dHacc, s.done, s.done + z.stripes, &sched, num_sms, st);
      }));
      void* out = static_cast<uint8_t*>(dH) + c0 * d * 2;
      FCKL_TRY(step(FCKL_K_OTHER, st, [&] { return launch_f32_to_bf16(s.dHacc, out, rows * d, st); }));
      continue;
    }
    for (int64_t s0 = 0; s0 < V; s0 += S) {
      const int64_t s_eff = (V - s0 < S) ? V - s0 : S;
      {
        const float* Hc = static_cast<const float*>(H) + c0 * d;
        const float* Wf = static_cast<const float*>(W);
        float* G = static_cast<float*>(s.G);
        FCKL_TRY(step(FCKL_K_BWD_TILES, st, [&] {
          return launch_simt_bwd_tiles(Hc, Wf, rows, d, V, s0, S, tau, s.sidx, s.sp, K, lse + c0, valid + c0, ctrl, G,
                                       st);
        }));
        FCKL_TRY(step(FCKL_K_GRAD_GEMM, st, [&] {
          return launch_simt_gemm(G, 1, S, Hc, d, 1, dW + s0 * d, d, s_eff, d, rows, c0 > 0, st);
        }));
        float* dHc = static_cast<float*>(dH) + c0 * d;
        FCKL_TRY(step(FCKL_K_GRAD_GEMM, st, [&] {
          return launch_simt_gemm(G, S, 1, Wf + s0 * d, d, 1, dHc, d, rows, d, s_eff, s0 > 0, st);
        }));
      }
    }
  }
  return FCKL_OK;
}

fckl_status fckl_topk_extract(const void* logits, int64_t T, int64_t V, int32_t K, fckl_dtype dtype,
                              int32_t* topk_idx, float* topk_logits, void* stream) {
  if (T < 0 || V < 1 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return FCKL_ERR_INVALID_ARG;
  if (K < 1 || K > FCKL_MAX_K || K > V) return FCKL_ERR_INVALID_ARG;
  if (dtype != FCKL_F32 && dtype != FCKL_BF16) return FCKL_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_idx || !topk_logits)) return FCKL_ERR_INVALID_ARG;
  if (!aligned(logits, dtype == FCKL_BF16 ? 2 : 4) || !aligned(topk_idx, 4) || !aligned(topk_logits, 4))
    return FCKL_ERR_UNSUPPORTED;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return step(FCKL_K_TOPK, st, [&] { return launch_topk(logits, T, V, K, dtype, topk_idx, topk_logits, st); });
}

fckl_status fckl_loss_partials(const void* ws, size_t ws_bytes, double* partials, void* stream) {
  if (!ws || !aligned(ws, kAlign) || ws_bytes < kCtrlBytes) return FCKL_ERR_WORKSPACE;
  if (!partials || !aligned(partials, 8)) return FCKL_ERR_INVALID_ARG;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Ctrl* ctrl = static_cast<const Ctrl*>(ws);
  return step(FCKL_K_REDUCE, st, [&] { return launch_loss_partials(ctrl, partials, st); });
}

fckl_status fckl_loss_finish(const double* total, const double* local, float* loss, float* grad_scale,
                             void* stream) {
  if (!total || !local || !loss || !grad_scale) return FCKL_ERR_INVALID_ARG;
  if (!aligned(total, 8) || !aligned(local, 8) || !aligned(loss, 4) || !aligned(grad_scale, 4))
    return FCKL_ERR_INVALID_ARG;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return step(FCKL_K_REDUCE, st, [&] { return launch_loss_finish(total, local, loss, grad_scale, st); });
}

fckl_status fckl_cast_f32_to_bf16(const float* src, void* dst, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!src || !dst))) return FCKL_ERR_INVALID_ARG;
  if (n % 4 != 0 || !aligned(src, 16) || !aligned(dst, 8)) return FCKL_ERR_UNSUPPORTED;
  if (n == 0) return FCKL_OK;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return step(FCKL_K_OTHER, st, [&] { return launch_f32_to_bf16(src, dst, n, st); });
}

fckl_status fckl_get_error(void* ws, void* stream) {
  if (!ws) return FCKL_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t status = 0;
  if (cudaMemcpyAsync(&status, ws, sizeof(status), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FCKL_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(status), st) != cudaSuccess) return FCKL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FCKL_ERR_CUDA;
  return static_cast<fckl_status>(status);
}

const char* fckl_status_string(fckl_status status) {
  switch (status) {
    case FCKL_OK: return "ok";
    case FCKL_ERR_INVALID_ARG: return "invalid argument (null pointer, size, K, tau or chunk out of range)";
    case FCKL_ERR_UNSUPPORTED: return "unsupported (alignment, d % 8 for bf16, or not an sm_103 device)";
    case FCKL_ERR_WORKSPACE: return "workspace null, too small or not 256-byte aligned";
    case FCKL_ERR_CUDA: return "a CUDA runtime call failed";
    case FCKL_ERR_BAD_INDEX: return "a teacher id lies outside [0, V)";
    case FCKL_ERR_TIMEOUT: return "an on-device wait timed out";
  }
  return "unknown status";
}

int64_t fckl_launch_count(void) { return g_launches.load(); }

void fckl_profile_enable(int on) { g_prof_on.store(on ? 1 : 0); }

fckl_status fckl_profile_read(int32_t kernel_class, int64_t* launches, double* total_ms, int reset) {
  if (kernel_class < 0 || kernel_class >= FCKL_K_NUM_CLASSES) return FCKL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (int c = 0; c < FCKL_K_NUM_CLASSES; ++c) {
    for (const Pending& p : g_pending[c]) {
      float ms = 0.f;
      if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
        return FCKL_ERR_CUDA;
      g_done_ms[c] += ms;
      g_done_launches[c] += 1;
      g_event_pool.push_back(p.a);
      g_event_pool.push_back(p.b);
    }
    g_pending[c].clear();
  }
  if (launches) *launches = g_done_launches[kernel_class];
  if (total_ms) *total_ms = g_done_ms[kernel_class];
  if (reset) {
    for (int c = 0; c < FCKL_K_NUM_CLASSES; ++c) {
      g_done_ms[c] = 0.0;
      g_done_launches[c] = 0;
    }
  }
  return FCKL_OK;
}

fckl_status fckl_debug_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, kAlign) || ws_bytes < kCtrlBytes) return FCKL_ERR_WORKSPACE;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);
  return step(FCKL_K_OTHER, st, [&] { return tc_debug_wait_timeout(ctrl, st); });
}

fckl_status fckl_debug_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K, int32_t a_mn,
                                 int32_t b_mn, int32_t cta_pair, void* stream) {
  if (!A || !B || !D || M < 1 || N < 1 || K < 1) return FCKL_ERR_INVALID_ARG;
  if (cta_pair && b_mn) return FCKL_ERR_UNSUPPORTED;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return FCKL_ERR_INVALID_ARG;
  if ((a_mn ? M : K) % 8 || (b_mn ? N : K) % 8 || N % 8) return FCKL_ERR_UNSUPPORTED;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16)) return FCKL_ERR_UNSUPPORTED;
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return step(FCKL_K_OTHER, st, [&] { return tc_debug_gemm(A, B, D, M, N, K, a_mn, b_mn, cta_pair, num_sms, st); });
}

}  // extern "C"
