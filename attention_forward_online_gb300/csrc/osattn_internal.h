// osattn_internal.h - launch interface between the C ABI (osattn_api.cu) and
// the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace osattn {

// Arguments of one forward call after host validation.
struct FwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* LSE;
  int B, H, Nq, Nkv, d;
  float scale;
  int causal;
  const int32_t* key_len;  // device, may be null
  cudaStream_t stream;
  unsigned int* status;    // device status word [0] and give-up site [1]
  uint64_t wait_limit_ns;
  int num_sms;
  // split-KV only (num_splits > 0): fp32 partials [num_splits, B*H, Nq, d]
  // and their LSE [num_splits, B*H, Nq]
  int num_splits = 0;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  int fp16 = 0;  // 16-bit element type: 0 bf16, 1 fp16
  // Element strides of the b, h and row axes (the d axis is contiguous).
  long long q_strides[3] = {0, 0, 0}, k_strides[3] = {0, 0, 0}, v_strides[3] = {0, 0, 0},
            o_strides[3] = {0, 0, 0};
};

// fp32 SIMT kernel (fwd_fp32_simt.cu).
cudaError_t launch_fwd_fp32(const FwdArgs& a);

// Tensor-core kernel for 16-bit inputs (fwd_bf16_tcgen05.cu).  The tensor
// maps describe Q, K and V as 4-D views (d, N, H, B) with the caller's
// strides and 128-byte swizzled 64 x 128 boxes.
cudaError_t prepare_fwd_bf16();  // once per device: kernel attributes
// Copies the forward kernel's per-step clock stamps (profiling builds) to
// host memory; *needed gets their size.  cudaErrorNotSupported otherwise.
cudaError_t read_step_trace(void* host, size_t bytes, size_t* needed);
cudaError_t launch_fwd_bf16(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV);

// Split-KV combine (splitkv_combine.cu): folds the partials of each row with
// the (m, l) combine and writes O (bf16) and LSE.
// Host checks of osattn_fwd_splitkv other than its workspace (pointers,
// sizes, alignment, scale, d, dtype, 1 <= num_splits <= OSATTN_MAX_SPLITS);
// OSATTN_OK or the status the entry point returns.
int validate_splitkv(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                     int B, int H, int Nq, int Nkv, int d, float scale, const int32_t* key_len,
                     int dtype, int num_splits);
cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* O,
                                   float* LSE, long long rows, int d, int num_splits, int fp16,
                                   cudaStream_t stream);

// Arguments of one backward call after host validation ([B, H, N, d]
// tensors with the strides below; 16-bit element type).
struct BwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const void* dO;
  const float* LSE;
  void* dQ;
  void* dK;
  void* dV;
  float* D;  // workspace [B, H, Nq]: rowsum(dO * O)
  int B, H, Nq, Nkv, d;
  float scale;
  int causal;
  const int32_t* key_len;  // device, may be null
  int fp16;                // 0 bf16, 1 fp16
  cudaStream_t stream;
  unsigned int* status;
  uint64_t wait_limit_ns;
  int num_sms;
  // Element strides of the b, h and row axes (the d axis is contiguous).
  long long q_strides[3], k_strides[3], v_strides[3], o_strides[3], do_strides[3],
      dq_strides[3], dk_strides[3], dv_strides[3];
};

// Backward kernels (bwd_tcgen05.cu): D = rowsum(dO * O), then dK/dV, then dQ.
cudaError_t prepare_bwd();  // once per device: kernel attributes
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmdO);
// fp32 path (bwd_fp32_simt.cu): D, then the SIMT dK/dV and dQ kernels.
cudaError_t prepare_bwd_fp32();  // once per device: kernel attributes
cudaError_t launch_bwd_fp32(const BwdArgs& a);
cudaError_t launch_bwd_rowdot_fp32(const BwdArgs& a);  // D for fp32 O and dO (bwd_tcgen05.cu)

// Standalone row softmax (softmax_rows.cu) over a [rows, N] matrix;
// elem: 0 bf16, 1 fp32, 2 fp16 (the public dtype codes).
// Row softmax: per-device set-up (cluster attributes; the largest cluster,
// 16 or 8 CTAs of 1024 threads, the GPU co-schedules) and the launch.
cudaError_t prepare_softmax_rows(int* max_cluster);
cudaError_t launch_softmax_rows(const void* in, void* out, float* lse, long long rows, int N,
                                int elem, int num_sms, int max_cluster, cudaStream_t stream);

// Box shape the bf16 kernel expects in its tensor maps.
constexpr int kBoxInner = 64;   // elements along d (128 bytes)
constexpr int kBoxRows = 128;   // rows of Q / K / V

}  // namespace osattn
