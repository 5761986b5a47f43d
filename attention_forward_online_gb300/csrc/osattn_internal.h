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
};

// fp32 SIMT kernel (fwd_fp32_simt.cu).
cudaError_t launch_fwd_fp32(const FwdArgs& a);

// bf16 tcgen05 kernel (fwd_bf16_tcgen05.cu).  The tensor maps describe Q, K
// and V as 3-D bf16 views (d, N, B*H) with 128-byte swizzled 64 x 128 boxes.
cudaError_t prepare_fwd_bf16();  // once per device: kernel attributes
cudaError_t launch_fwd_bf16(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV);

// Split-KV combine (splitkv_combine.cu): folds the partials of each row with
// the (m, l) combine and writes O (bf16) and LSE.
cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* O,
                                   float* LSE, long long rows, int d, int num_splits,
                                   cudaStream_t stream);

// Standalone row softmax (softmax_rows.cu) over a [rows, N] matrix.
cudaError_t launch_softmax_rows(const void* in, void* out, float* lse, long long rows, int N,
                                int dtype_fp32, int num_sms, cudaStream_t stream);

// Box shape the bf16 kernel expects in its tensor maps.
constexpr int kBoxInner = 64;   // elements along d (128 bytes)
constexpr int kBoxRows = 128;   // rows of Q / K / V

}  // namespace osattn
