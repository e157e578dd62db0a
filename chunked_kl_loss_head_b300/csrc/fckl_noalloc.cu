// fckl_noalloc.cu -- fckl_forward_noalloc: the forward pass for callers that cannot
// allocate device memory (see include/fckl.h).  Its scratch is a fixed array in this
// library's own device memory instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "fckl_internal.h"

namespace fckl {
namespace {

// The scratch every call of fckl_forward_noalloc uses.  It lives as long as the library
// is loaded, on every GPU that loads it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FCKL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  Host code cannot use the
// symbol itself (on the host it names a stand-in, not device memory), so the address is
// looked up once per device with that device current and kept.
fckl_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FCKL_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FCKL_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FCKL_OK;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Scratch bytes of one chunk of `rows` rows.
size_t chunk_bytes(int64_t rows, int64_t K, int64_t nvt) {
  const size_t ck = static_cast<size_t>(rows) * static_cast<size_t>(K);
  return up256(sizeof(Ctrl)) + 4 * up256(4 * ck) + up256(8 * static_cast<size_t>(rows) * static_cast<size_t>(nvt));
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace fckl

using namespace fckl;

extern "C" fckl_status fckl_forward_noalloc(const void* H, const void* W, const int32_t* topk_idx,
                                            const float* topk_logits, const uint8_t* valid, int64_t T, int64_t d,
                                            int64_t V, int32_t K, float tau, int64_t chunk, fckl_dtype dtype,
                                            float* loss, float* lse, float* row_loss, int32_t* status,
                                            void* stream) {
  // ---- argument checks (nothing is launched or looked up before they pass)
  if (T < 0 || d < 1 || V < 1 || K < 1 || K > FCKL_MAX_K || chunk < 1) return FCKL_ERR_INVALID_ARG;
  if (dtype != FCKL_F32 && dtype != FCKL_BF16) return FCKL_ERR_INVALID_ARG;
  if (V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || d >= (int64_t(1) << 31)) return FCKL_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !std::isfinite(tau)) return FCKL_ERR_INVALID_ARG;
  if (!loss) return FCKL_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !topk_idx || !topk_logits || !valid || !lse || !row_loss)) return FCKL_ERR_INVALID_ARG;
  if (!is_aligned(topk_idx, 4) || !is_aligned(topk_logits, 4)) return FCKL_ERR_UNSUPPORTED;
  if (dtype == FCKL_BF16 ? (d % 8 != 0 || !is_aligned(H, 16) || !is_aligned(W, 16))
                         : (!is_aligned(H, 4) || !is_aligned(W, 4)))
    return FCKL_ERR_UNSUPPORTED;
  const int64_t nvt = (V + kTileV - 1) / kTileV;
  // the largest chunk that fits the fixed scratch (a multiple of 128 rows when possible);
  // the result does not depend on the chunk size
  int64_t rows_max = chunk < T ? chunk : (T > 0 ? T : 1);
  if (chunk_bytes(1, K, nvt) > FCKL_NOALLOC_SCRATCH_BYTES) return FCKL_ERR_WORKSPACE;
  while (rows_max > 1 && chunk_bytes(rows_max, K, nvt) > FCKL_NOALLOC_SCRATCH_BYTES) {
    rows_max = rows_max > 256 ? (rows_max - 1) / 128 * 128 : rows_max / 2;
  }

  // ---- device and scratch
  int dev = 0, major = 0, minor = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FCKL_ERR_CUDA;
  if (major != 10 || minor != 3) return FCKL_ERR_UNSUPPORTED;
  void* base = nullptr;
  const fckl_status sa = scratch_address(&base);
  if (sa != FCKL_OK) return sa;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  uint8_t* b = static_cast<uint8_t*>(base);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(b);
  size_t off = up256(sizeof(Ctrl));
  const size_t ck = static_cast<size_t>(rows_max) * static_cast<size_t>(K);
  ChunkScratch s{};
  s.sidx = reinterpret_cast<int32_t*>(b + off);
  off += up256(4 * ck);
  s.sp = reinterpret_cast<float*>(b + off);
  off += up256(4 * ck);
  s.slogp = reinterpret_cast<float*>(b + off);
  off += up256(4 * ck);
  s.zk = reinterpret_cast<float*>(b + off);
  off += up256(4 * ck);
  s.part = reinterpret_cast<float2*>(b + off);

  // the previous call's status word must not leak into this one
  if (cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st) != cudaSuccess) return FCKL_ERR_CUDA;
  TileSched sched{&ctrl->tile_counter, 0};
  const int nv = static_cast<int>(nvt);
  for (int64_t c0 = 0; c0 < T; c0 += rows_max) {
    const int64_t rows = (T - c0 < rows_max) ? T - c0 : rows_max;
    if (launch_prep(topk_idx + c0 * K, topk_logits + c0 * K, rows, K, V, tau, s, ctrl, st) != cudaSuccess)
      return FCKL_ERR_CUDA;
    count_launch(FCKL_K_PREP);
    cudaError_t e;
    if (dtype == FCKL_BF16) {
      e = tc_fwd_tiles(static_cast<const uint8_t*>(H) + c0 * d * 2, W, rows, d, V, tau, s.sidx, K, s.zk, s.part, nv,
                       ctrl, &sched, num_sms, st);
    } else {
      e = launch_simt_fwd_tiles(static_cast<const float*>(H) + c0 * d, static_cast<const float*>(W), rows, d, V, tau,
                                s.sidx, K, s.zk, s.part, nv, st);
    }
    if (e != cudaSuccess) return FCKL_ERR_CUDA;
    count_launch(FCKL_K_FWD_TILES);
    if (launch_combine(s.part, nv, s.zk, s.sp, s.slogp, valid + c0, rows, K, tau, lse + c0, row_loss + c0, st) !=
        cudaSuccess)
      return FCKL_ERR_CUDA;
    count_launch(FCKL_K_COMBINE);
  }
  if (launch_loss_reduce(row_loss, valid, T, loss, ctrl, st) != cudaSuccess) return FCKL_ERR_CUDA;
  count_launch(FCKL_K_REDUCE);
  if (status && cudaMemcpyAsync(status, &ctrl->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return FCKL_ERR_CUDA;
  return FCKL_OK;
}
