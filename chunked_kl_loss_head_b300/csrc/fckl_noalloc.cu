// fckl_noalloc.cu -- fckl_forward_noalloc: the forward pass for callers that cannot
// allocate device memory (see include/fckl.h).  Its scratch is a fixed array in this
// library's own device memory instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <cmath>

#include "fckl_internal.h"

namespace fckl {
namespace {

// The scratch every call of fckl_forward_noalloc uses.  It lives as long as the library
// is loaded, on every GPU that loads it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FCKL_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  Host code cannot use the
// symbol itself (on the host it names a stand-in, not device memory), so the address is
// looked up with that device current, on every call: the lookup is cheap once the
// library's GPU code is loaded, and an address kept from an earlier call would go stale
// if the device's context were torn down and the code loaded again elsewhere.
fckl_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FCKL_ERR_CUDA;
  *out = p;
  return FCKL_OK;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Scratch bytes of one chunk of `rows` rows.
size_t chunk_bytes(int64_t rows, int64_t K, int64_t nvt) {
  const size_t ck = static_cast<size_t>(rows) * static_cast<size_t>(K);
  return up256(sizeof(Ctrl)) + 4 * up256(4 * ck) + up256(8 * static_cast<size_t>(rows) * static_cast<size_t>(nvt));
}

}  // namespace
}  // namespace fckl

using namespace fckl;

extern "C" fckl_status fckl_forward_noalloc(const void* H, const void* W, const int32_t* topk_idx,
                                            const float* topk_logits, const uint8_t* valid, int64_t T, int64_t d,
                                            int64_t V, int32_t K, float tau, int64_t chunk, fckl_dtype dtype,
                                            float* loss, float* lse, float* row_loss, int32_t* status,
                                            void* stream) {
  // ---- argument checks (nothing is launched or looked up before they pass)
  if (!valid_sizes(T, d, V, K, chunk, dtype)) return FCKL_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !std::isfinite(tau)) return FCKL_ERR_INVALID_ARG;
  if (!loss) return FCKL_ERR_INVALID_ARG;
  if (T > 0 && (!H || !W || !topk_idx || !topk_logits || !valid || !lse || !row_loss)) return FCKL_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(topk_logits, 4)) return FCKL_ERR_UNSUPPORTED;
  if (dtype == FCKL_BF16 ? (d % 8 != 0 || !aligned(H, 16) || !aligned(W, 16)) : (!aligned(H, 4) || !aligned(W, 4)))
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
  int num_sms = 0;
  FCKL_TRY(device_info(&num_sms));
  void* base = nullptr;
  FCKL_TRY(scratch_address(&base));
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

  // the previous call's status word and tile counter must not leak into this one
  FCKL_TRY(step(FCKL_K_OTHER, st, [&] { return cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st); }));
  TileSched sched{&ctrl->tile_counter, 0};
  const int nv = static_cast<int>(nvt);
  for (int64_t c0 = 0; c0 < T; c0 += rows_max) {
    const int64_t rows = (T - c0 < rows_max) ? T - c0 : rows_max;
    FCKL_TRY(step(FCKL_K_PREP, st, [&] {
      return launch_prep(topk_idx + c0 * K, topk_logits + c0 * K, rows, K, V, tau, s, ctrl, st);
    }));
    FCKL_TRY(step(FCKL_K_FWD_TILES, st, [&] {
      if (dtype == FCKL_BF16)
        return tc_fwd_tiles(static_cast<const uint8_t*>(H) + c0 * d * 2, W, rows, d, V, tau, s.sidx, K, s.zk,
                            s.part, nv, ctrl, &sched, num_sms, st);
      return launch_simt_fwd_tiles(static_cast<const float*>(H) + c0 * d, static_cast<const float*>(W), rows, d, V,
                                   tau, s.sidx, K, s.zk, s.part, nv, st);
    }));
    FCKL_TRY(step(FCKL_K_COMBINE, st, [&] {
      return launch_combine(s.part, nv, s.zk, s.sp, s.slogp, valid + c0, rows, K, tau, lse + c0, row_loss + c0, st);
    }));
  }
  FCKL_TRY(step(FCKL_K_REDUCE, st, [&] { return launch_loss_reduce(row_loss, valid, T, loss, ctrl, st); }));
  if (status) {
    FCKL_TRY(step(FCKL_K_OTHER, st, [&] {
      return cudaMemcpyAsync(status, &ctrl->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    }));
  }
  return FCKL_OK;
}
