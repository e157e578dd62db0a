// fckl_internal.h -- declarations shared by the host API and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fckl.h"

namespace fckl {

constexpr int kTileM = 128;   // rows (tokens) of one logit tile
constexpr int kTileV = 256;   // vocab columns of one logit tile (forward partial granularity)
constexpr int kCtrlBytes = 256;

// First bytes of the workspace: status word and scalars shared between kernels.
struct Ctrl {
  int32_t status;        // first device-detected fckl_status (0 = none)
  int32_t pad0;
  int64_t n_valid;       // N of the last reduction
  float grad_alpha;      // g / (tau * N) for the backward (0 when N = 0)
  float pad1;
  double loss_sum;       // sum of valid loss_t of the last forward
  uint32_t tile_counter; // dynamic tile scheduler of the tensor-core launches
  uint32_t pad2;
};

// Host-side view of the tile counter: its device address and the value it will hold when
// the next launch on the stream starts.
struct TileSched {
  unsigned int* counter;
  unsigned int value;
};

// Records `code` as the workspace status unless one is already recorded.
__device__ __forceinline__ void set_status(Ctrl* ctrl, int code) {
  atomicCAS(&ctrl->status, 0, code);
}

// Per-chunk scratch carved out of the workspace.
struct ChunkScratch {
  int32_t* sidx;    // [C, K] teacher ids of each row, ascending (bad ids -> INT32_MAX)
  float* sp;        // [C, K] teacher p, permuted like sidx
  float* slogp;     // [C, K] teacher log p, permuted like sidx
  float* zk;        // [C, K] student logit at sidx (forward)
  float2* part;     // [C, nvt] per (row, 256-wide vocab tile): (max, sum) in log2 units
  void* G;          // gradient stripes: [C, 3 S] bf16 (bf16 work) or [C, S] f32 (f32 work)
  unsigned int* done;  // [2, stripes] completion counters of the chunk backward (bf16 work)
  float* dHacc;     // [C, d] fp32 dH accumulator (bf16 work only)
  void* HcT;        // [d, ldT] bf16 transposed hidden states of the chunk (bf16 work only)
  int64_t ldT;      // C rounded up to a multiple of 8
};

// ---- row kernels (fckl_rowops.cu) --------------------------------------------------------
cudaError_t launch_prep(const int32_t* idx, const float* logits, int64_t rows, int32_t K, int64_t V,
                        float tau, ChunkScratch s, Ctrl* ctrl, cudaStream_t st);
cudaError_t launch_combine(const float2* part, int nvt, const float* zk, const float* sp,
                           const float* slogp, const uint8_t* valid, int64_t rows, int32_t K,
                           float tau, float* lse, float* row_loss, cudaStream_t st);
cudaError_t launch_loss_reduce(const float* row_loss, const uint8_t* valid, int64_t T, float* loss,
                               Ctrl* ctrl, cudaStream_t st);
cudaError_t launch_grad_scale(const uint8_t* valid, int64_t T, float tau, float grad_loss,
                              const float* grad_scale, Ctrl* ctrl, cudaStream_t st);
cudaError_t launch_loss_partials(const Ctrl* ctrl, double* out, cudaStream_t st);
cudaError_t launch_loss_finish(const double* total, const double* local, float* loss, float* grad_scale,
                               cudaStream_t st);
cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t st);
// out[c, r] = in[r, c] for bf16 in[rows, cols] (row stride ld_in) -> out[cols, ld_out]
cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out,
                                  int64_t ld_out, cudaStream_t st);

// ---- teacher top-K extraction (fckl_topk.cu) ----------------------------------------------
cudaError_t launch_topk(const void* logits, int64_t T, int64_t V, int32_t K, fckl_dtype dtype,
                        int32_t* idx, float* val, cudaStream_t st);

// ---- fp32 CUDA-core path (fckl_simt.cu) --------------------------------------------------
cudaError_t launch_simt_fwd_tiles(const float* Hc, const float* W, int64_t rows, int64_t d, int64_t V,
                                  float tau, const int32_t* sidx, int32_t K, float* zk, float2* part,
                                  int nvt, cudaStream_t st);
cudaError_t launch_simt_bwd_tiles(const float* Hc, const float* W, int64_t rows, int64_t d, int64_t V,
                                  int64_t s0, int64_t S, float tau, const int32_t* sidx,
                                  const float* sp, int32_t K, const float* lse, const uint8_t* valid,
                                  const Ctrl* ctrl, float* G, cudaStream_t st);
// C[M, N] = beta * C + sum_k A(m, k) B(k, n), A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn]
cudaError_t launch_simt_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk,
                             int64_t sbn, float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             int beta, cudaStream_t st);

// ---- bf16 tensor-core path (fckl_tc.cu) --------------------------------------------------
cudaError_t tc_fwd_tiles(const void* Hc, const void* W, int64_t rows, int64_t d, int64_t V,
                         float tau, const int32_t* sidx, int32_t K, float* zk, float2* part, int nvt,
                         Ctrl* ctrl, TileSched* sched, int num_sms, cudaStream_t st);
// Gradient buffers the chunk backward rotates through (each [rows, S] bf16, side by side).
int tc_grad_buffers();
// The whole backward of one chunk in one launch, over every vocab stripe of width S:
//   G_s = (softmax - p) * g / (tau N) of the recomputed logit tile H_chunk . W_s^T (bf16)
//   dH accumulator acc[rows, d] += G_s . W_s            (acc must hold zeros at entry)
//   dW[s*S:(s+1)*S, :] (+)= G_s^T . H_chunk             (stored when !dW_accumulate)
// G is [rows, 3 S] bf16 (three rotating stripe buffers); HcT is H_chunk transposed, [d, ldT]
// bf16; done_g / done_w are [ceil(V / S)] completion counters that must hold zeros at entry.
cudaError_t tc_bwd_chunk(const void* Hc, const void* HcT, int64_t ldT, const void* W, int64_t rows,
                         int64_t d, int64_t V, int64_t S, float tau, const int32_t* sidx,
                         const float* sp, int32_t K, const float* lse, const uint8_t* valid,
                         Ctrl* ctrl, void* G, float* dW, int dW_accumulate, float* dH_acc,
                         unsigned int* done_g, unsigned int* done_w, TileSched* sched, int num_sms,
                         cudaStream_t st);
cudaError_t tc_debug_wait_timeout(Ctrl* ctrl, cudaStream_t st);
cudaError_t tc_debug_gemm(const void* A, const void* B, float* D, int64_t M, int64_t N, int64_t K,
                          int a_mn, int b_mn, int cta_pair, int num_sms, cudaStream_t st);

// ---- host helpers (fckl_api.cu) ----------------------------------------------------------
// Size arguments every loss entry point shares: T >= 0, d, V >= 1, 1 <= K <= FCKL_MAX_K,
// chunk >= 1, a known dtype, and T, d, V below 2^31.
bool valid_sizes(int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, fckl_dtype dt);
// Device check (the kernels are built for sm_103a only) and the SM count of the current
// device.
fckl_status device_info(int* num_sms);
bool aligned(const void* p, size_t a);
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
bool encode_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
void count_launch(fckl_kernel_class cls);
void prof_begin(fckl_kernel_class cls, cudaStream_t st);
void prof_end(fckl_kernel_class cls, cudaStream_t st);

// Runs one launch step: counts it, brackets it with events when profiling is on, and maps a
// CUDA error to FCKL_ERR_CUDA.
template <class F>
fckl_status step(fckl_kernel_class cls, cudaStream_t st, F&& launch) {
  prof_begin(cls, st);
  const cudaError_t e = launch();
  prof_end(cls, st);
  if (e != cudaSuccess) return FCKL_ERR_CUDA;
  count_launch(cls);
  return FCKL_OK;
}

#define FCKL_TRY(expr)             \
  do {                             \
    const fckl_status _s = (expr); \
    if (_s != FCKL_OK) return _s;  \
  } while (0)

}  // namespace fckl
