// osattn_api.cu - the C ABI of libosattn (declared in include/osattn.h):
// argument validation, per-device set-up, TMA descriptor encoding and kernel
// selection.  Every step of the computation runs in the CUDA kernels; this
// file only checks arguments and enqueues them.
#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "osattn.h"
#include "osattn_internal.h"
#include "sm100_ptx.cuh"

namespace {

// Device status: [0] = OSATTN_OK or OSATTN_ERR_TIMEOUT, [1] = site of the
// first wait that gave up.  One copy per device that loads the library.
__device__ unsigned int g_device_status[2];

constexpr int kMaxDevices = 64;

constexpr int kOffloadEvents = 64;  // event ring of the offload pipeline

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int row_cluster_max = 8;  // CTAs per cluster of the split-row softmax
  unsigned int* status = nullptr;  // device address of g_device_status
  // Offload pipeline (osattn_fwd_offload), created on first use: a
  // host-to-device and a device-to-host copy stream, a second compute
  // stream, and their events.
  bool offload_ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, cmp = nullptr;
  cudaEvent_t ev_entry = nullptr, ev_final = nullptr;
  cudaEvent_t ev_in[kOffloadEvents] = {}, ev_out[kOffloadEvents] = {};
};

std::mutex g_offload_mutex;  // one offload enqueue at a time (shared streams and events)

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{4000000000ull};
std::atomic<int> g_last_timeout_site{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_tiled = nullptr;

// Per-device set-up, done once with the device current: SM count, the
// device address of the status word, kernel attributes, and the driver's
// tensor-map encoder.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return OSATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OSATTN_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_device_status) !=
        cudaSuccess)
      return OSATTN_ERR_CUDA;
    if (osattn::prepare_fwd_bf16() != cudaSuccess) return OSATTN_ERR_CUDA;
    if (osattn::prepare_bwd() != cudaSuccess || osattn::prepare_bwd_fp32() != cudaSuccess)
      return OSATTN_ERR_CUDA;
    if (osattn::prepare_softmax_rows(&st.row_cluster_max) != cudaSuccess) return OSATTN_ERR_CUDA;
    if (!g_encode_tiled) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return OSATTN_ERR_CUDA;
      g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return OSATTN_OK;
}

// 4-D view (d, N, H, B) of a tensor with element strides st = {b, h, row}
// (d contiguous), 64 x 128 boxes, 128-byte swizzle, zero fill outside it.
int encode_map(CUtensorMap* map, const void* base, int fp16, int d, int N, int H, int B,
               const long long* st) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2,
                                 static_cast<cuuint64_t>(st[1]) * 2,
                                 static_cast<cuuint64_t>(st[0]) * 2};
  const cuuint32_t box[4] = {osattn::kBoxInner, osattn::kBoxRows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode_tiled(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OSATTN_OK : OSATTN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

__global__ void wait_timeout_kernel(unsigned int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    osattn::mbar_init(&bar, 1);
    abort_flag = 0;
    osattn::fence_barrier_init();
  }
  __syncwarp();
  // Nobody arrives on `bar`: the wait must give up after limit_ns.
  const osattn::WaitCtl wc{&abort_flag, status, status + 1, limit_ns};
  osattn::mbar_wait(&bar, 0, wc, 99u);
}

}  // namespace

extern "C" {

int osattn_version(void) { return OSATTN_VERSION; }

const char* osattn_status_string(int status) {
  switch (status) {
    case OSATTN_OK: return "ok";
    case OSATTN_ERR_INVALID_ARG: return "invalid argument";
    case OSATTN_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case OSATTN_ERR_CUDA: return "CUDA error";
    case OSATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case OSATTN_ERR_SCRATCH_LIMIT:
      return "problem needs more split-KV scratch than the library's built-in array";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

size_t elem_size(int dtype) { return dtype == OSATTN_FP32 ? 4 : 2; }

// Host validation shared by every forward entry point; nothing is enqueued
// when it fails.
int validate_fwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                 int B, int H, int Nq, int Nkv, int d, float scale, const int32_t* key_len,
                 int dtype) {
  if (!Q || !K || !V || !O || !LSE) return OSATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nkv < 1 || d < 1) return OSATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return OSATTN_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
      !aligned(LSE, 4) || (key_len && !aligned(key_len, 4)))
    return OSATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return OSATTN_ERR_UNSUPPORTED;
  if (dtype != OSATTN_BF16 && dtype != OSATTN_FP32 && dtype != OSATTN_FP16)
    return OSATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return OSATTN_ERR_INVALID_ARG;
  return OSATTN_OK;
}

// Element strides {b, h, row}: the caller's, or those of a contiguous
// [B, H, N, d] tensor when `in` is null.  Every stride must be >= 1 and keep
// each row 16-byte aligned (a multiple of 16 bytes) and below 2^40 bytes.
int take_strides(const int64_t* in, int H, int N, int d, int dtype, long long* out) {
  if (!in) {
    out[2] = d;
    out[1] = static_cast<long long>(N) * d;
    out[0] = static_cast<long long>(H) * N * d;
    return OSATTN_OK;
  }
  const long long es = static_cast<long long>(elem_size(dtype));
  for (int i = 0; i < 3; ++i) {
    if (in[i] < 1 || (in[i] * es) % 16 != 0 || in[i] * es >= (1LL << 40))
      return OSATTN_ERR_INVALID_ARG;
    out[i] = in[i];
  }
  return OSATTN_OK;
}

osattn::FwdArgs make_args(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                          int H, int Nq, int Nkv, int d, float scale, int causal,
                          const int32_t* key_len, void* stream, const DeviceState* st) {
  osattn::FwdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.LSE = LSE;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nkv = Nkv;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.key_len = key_len;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = st->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.num_sms = st->num_sms;
  return a;
}

int encode_qkv(const osattn::FwdArgs& a, CUtensorMap* tmQ, CUtensorMap* tmK, CUtensorMap* tmV) {
  if (encode_map(tmQ, a.Q, a.fp16, a.d, a.Nq, a.H, a.B, a.q_strides) != OSATTN_OK ||
      encode_map(tmK, a.K, a.fp16, a.d, a.Nkv, a.H, a.B, a.k_strides) != OSATTN_OK ||
      encode_map(tmV, a.V, a.fp16, a.d, a.Nkv, a.H, a.B, a.v_strides) != OSATTN_OK)
    return OSATTN_ERR_CUDA;
  return OSATTN_OK;
}

// Split-KV launch over caller-provided partial buffers: the key-range split
// of the tensor-core kernel, then the combine.  Arguments are validated.
int launch_splitkv(osattn::FwdArgs a, int num_splits, float* o_part, float* lse_part) {
  CUtensorMap tmQ, tmK, tmV;
  if (encode_qkv(a, &tmQ, &tmK, &tmV) != OSATTN_OK) return OSATTN_ERR_CUDA;
  a.num_splits = num_splits;
  a.o_part = o_part;
  a.lse_part = lse_part;
  if (osattn::launch_fwd_bf16(a, tmQ, tmK, tmV) != cudaSuccess) return OSATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  if (osattn::launch_splitkv_combine(o_part, lse_part, a.O, a.LSE, rows, a.d, num_splits, a.fp16,
                                     a.stream) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  return OSATTN_OK;
}

int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
             int Nq, int Nkv, int d, const int64_t* q_strides, const int64_t* k_strides,
             const int64_t* v_strides, const int64_t* o_strides, float scale, int causal,
             const int32_t* key_len, int dtype, void* stream) {
  int rc = validate_fwd(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, key_len, dtype);
  if (rc != OSATTN_OK) return rc;
  long long qs[3], ks[3], vs[3], os[3];
  if (take_strides(q_strides, H, Nq, d, dtype, qs) != OSATTN_OK ||
      take_strides(k_strides, H, Nkv, d, dtype, ks) != OSATTN_OK ||
      take_strides(v_strides, H, Nkv, d, dtype, vs) != OSATTN_OK ||
      take_strides(o_strides, H, Nq, d, dtype, os) != OSATTN_OK)
    return OSATTN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != OSATTN_OK) return rc;
  osattn::FwdArgs a = make_args(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, causal, key_len, stream, st);
  for (int i = 0; i < 3; ++i) {
    a.q_strides[i] = qs[i];
    a.k_strides[i] = ks[i];
    a.v_strides[i] = vs[i];
    a.o_strides[i] = os[i];
  }
  cudaError_t e;
  if (dtype == OSATTN_FP32) {
    e = osattn::launch_fwd_fp32(a);
  } else {
    a.fp16 = dtype == OSATTN_FP16;
    CUtensorMap tmQ, tmK, tmV;
    if (encode_qkv(a, &tmQ, &tmK, &tmV) != OSATTN_OK) return OSATTN_ERR_CUDA;
    e = osattn::launch_fwd_bf16(a, tmQ, tmK, tmV);
  }
  return e == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
}

int offload_streams(DeviceState* ds) {
  if (ds->offload_ready) return OSATTN_OK;
  const unsigned ef = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&ds->h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ds->d2h, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ds->cmp, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ds->ev_entry, ef) != cudaSuccess ||
      cudaEventCreateWithFlags(&ds->ev_final, ef) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  for (int i = 0; i < kOffloadEvents; ++i)
    if (cudaEventCreateWithFlags(&ds->ev_in[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&ds->ev_out[i], ef) != cudaSuccess)
      return OSATTN_ERR_CUDA;
  ds->offload_ready = true;
  return OSATTN_OK;
}

// One tensor of an offload pipeline: host and device copies of a
// contiguous [B, H, ...] tensor and the bytes of one head.
struct OffloadSeg {
  void* host;
  void* dev;
  size_t head_bytes;
};

// Host -> device -> host pipeline over chunks of heads: the copy of chunk
// c + 1 in, the compute of chunk c and the copy of chunk c - 1 out run
// concurrently on the library's two copy streams and the compute streams.
// With `alternate`, chunks alternate between the caller's stream and the
// library's second compute stream, so that a chunk's launch can start on
// the SMs the tail of the previous one leaves idle (for work whose chunks
// touch disjoint parts of every buffer); otherwise all run on the caller's
// stream.  compute(b, h0, nh, s) enqueues the work of heads
// h0 .. h0 + nh - 1 of batch entry b on stream s.
template <typename Compute>
int offload_enqueue(DeviceState* ds, cudaStream_t cs, int B, int H, int hc, const OffloadSeg* ins,
                    int n_in, const OffloadSeg* outs, int n_out, bool alternate, Compute&& compute) {
  int rc = OSATTN_OK;
  // Copies wait for the caller's earlier work on `stream` (it may still be
  // reading the device buffers).
  if (cudaEventRecord(ds->ev_entry, cs) != cudaSuccess ||
      cudaStreamWaitEvent(ds->h2d, ds->ev_entry, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ds->d2h, ds->ev_entry, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ds->cmp, ds->ev_entry, 0) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  int c = 0;
  for (int b = 0; b < B; ++b) {
    for (int h0 = 0; h0 < H; h0 += hc, ++c) {
      const int nh = H - h0 < hc ? H - h0 : hc;
      const size_t head0 = static_cast<size_t>(b) * H + h0;
      cudaEvent_t ein = ds->ev_in[c % kOffloadEvents], eout = ds->ev_out[c % kOffloadEvents];
      for (int i = 0; i < n_in; ++i) {
        const size_t off = head0 * ins[i].head_bytes;
        if (cudaMemcpyAsync(static_cast<char*>(ins[i].dev) + off,
                            static_cast<const char*>(ins[i].host) + off, nh * ins[i].head_bytes,
                            cudaMemcpyHostToDevice, ds->h2d) != cudaSuccess)
          return OSATTN_ERR_CUDA;
      }
      const cudaStream_t ks = (alternate && (c & 1)) ? ds->cmp : cs;
      if (cudaEventRecord(ein, ds->h2d) != cudaSuccess || cudaStreamWaitEvent(ks, ein, 0) != cudaSuccess)
        return OSATTN_ERR_CUDA;
      rc = compute(b, h0, nh, ks);
      if (rc != OSATTN_OK) return rc;
      if (cudaEventRecord(eout, ks) != cudaSuccess || cudaStreamWaitEvent(ds->d2h, eout, 0) != cudaSuccess)
        return OSATTN_ERR_CUDA;
      for (int i = 0; i < n_out; ++i) {
        const size_t off = head0 * outs[i].head_bytes;
        if (cudaMemcpyAsync(static_cast<char*>(outs[i].host) + off,
                            static_cast<const char*>(outs[i].dev) + off, nh * outs[i].head_bytes,
                            cudaMemcpyDeviceToHost, ds->d2h) != cudaSuccess)
          return OSATTN_ERR_CUDA;
      }
    }
  }
  return OSATTN_OK;
}

// offload_enqueue under the offload mutex (the copy streams and events are
// shared), with both copy streams joined back into `stream` on every exit.
template <typename Compute>
int offload_pipeline(DeviceState* ds, cudaStream_t cs, int B, int H, int hc, const OffloadSeg* ins,
                     int n_in, const OffloadSeg* outs, int n_out, bool alternate,
                     Compute&& compute) {
  std::lock_guard<std::mutex> lock(g_offload_mutex);
  int rc = offload_streams(ds);
  if (rc != OSATTN_OK) return rc;
  rc = offload_enqueue(ds, cs, B, H, hc, ins, n_in, outs, n_out, alternate, compute);
  // `stream` completes only after the last copy, in either direction, and
  // the last compute on the second stream, even when the enqueue stopped
  // part way (the caller may free the buffers once `stream` is done).
  bool joined = true;
  for (cudaStream_t cp : {ds->h2d, ds->d2h, ds->cmp})
    joined = joined && cudaEventRecord(ds->ev_final, cp) == cudaSuccess &&
             cudaStreamWaitEvent(cs, ds->ev_final, 0) == cudaSuccess;
  if (rc != OSATTN_OK) return rc;
  return joined ? OSATTN_OK : OSATTN_ERR_CUDA;
}

// Heads per chunk: the caller's, or (0) enough that a chunk's launch covers
// `waves` waves of CTAs of `rows_per_cta` rows out of N.
int offload_heads(int heads_per_chunk, int H, int N, int rows_per_cta, int num_sms, int waves) {
  long long hc = heads_per_chunk;
  if (hc == 0) {
    const long long units = (N + rows_per_cta - 1) / rows_per_cta;
    hc = (static_cast<long long>(waves) * num_sms + units - 1) / units;
  }
  return static_cast<int>(hc < H ? hc : H);
}

int fwd_offload_impl(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh,
                     void* Qd, void* Kd, void* Vd, void* Od, float* LSEd, int B, int H, int Nq,
                     int Nkv, int d, float scale, int causal, const int32_t* key_len, int dtype,
                     int heads_per_chunk, void* stream) {
  if (!Qh || !Kh || !Vh || !Oh || !LSEh) return OSATTN_ERR_INVALID_ARG;
  int rc = validate_fwd(Qd, Kd, Vd, Od, LSEd, B, H, Nq, Nkv, d, scale, key_len, dtype);
  if (rc != OSATTN_OK) return rc;
  if (heads_per_chunk < 0) return OSATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  rc = device_state(&ds);
  if (rc != OSATTN_OK) return rc;
  // 256 query rows per CTA on the tensor cores, 16 in the fp32 kernel; one
  // wave of CTAs a chunk (consecutive chunks overlap on two compute streams:
  // on causal B1 H32 16K d128 from pinned host memory, 2.43 ms a call with
  // 3-head chunks against 2.52 with 5)
  const int hc = offload_heads(heads_per_chunk, H, Nq, dtype == OSATTN_FP32 ? 16 : 256, ds->num_sms,
                               1);
  const size_t es = elem_size(dtype);
  const size_t qb = static_cast<size_t>(Nq) * d * es, kb = static_cast<size_t>(Nkv) * d * es;
  const size_t lb = static_cast<size_t>(Nq) * sizeof(float);
  const OffloadSeg ins[3] = {{const_cast<void*>(Qh), Qd, qb}, {const_cast<void*>(Kh), Kd, kb},
                             {const_cast<void*>(Vh), Vd, kb}};
  const OffloadSeg outs[2] = {{Oh, Od, qb}, {LSEh, LSEd, lb}};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return offload_pipeline(ds, cs, B, H, hc, ins, 3, outs, 2, true, [&](int b, int h0, int nh,
                                                                cudaStream_t ks) {
    const size_t head0 = static_cast<size_t>(b) * H + h0;
    return fwd_impl(static_cast<const char*>(Qd) + head0 * qb, static_cast<const char*>(Kd) + head0 * kb,
                    static_cast<const char*>(Vd) + head0 * kb, static_cast<char*>(Od) + head0 * qb,
                    LSEd + head0 * Nq, 1, nh, Nq, Nkv, d, nullptr, nullptr, nullptr, nullptr, scale,
                    causal, key_len ? key_len + b : nullptr, dtype, ks);
  });
}

int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nkv, int d,
             const int64_t* const* strides, float scale, int causal, const int32_t* key_len,
             int dtype, void* workspace, size_t workspace_bytes, void* stream);

int bwd_offload_impl(const void* Qh, const void* Kh, const void* Vh, const void* Oh,
                     const void* dOh, const float* LSEh, void* dQh, void* dKh, void* dVh, void* Qd,
                     void* Kd, void* Vd, void* Od, void* dOd, float* LSEd, void* dQd, void* dKd,
                     void* dVd, int B, int H, int Nq, int Nkv, int d, float scale, int causal,
                     const int32_t* key_len, int dtype, void* workspace, size_t workspace_bytes,
                     int heads_per_chunk, void* stream) {
  if (!Qh || !Kh || !Vh || !Oh || !dOh || !LSEh || !dQh || !dKh || !dVh)
    return OSATTN_ERR_INVALID_ARG;
  // Argument checks of osattn_bwd on the whole tensors, before any copy.
  int rc = validate_fwd(Qd, Kd, Vd, Od, LSEd, B, H, Nq, Nkv, d, scale, key_len, dtype);
  if (rc != OSATTN_OK) return rc;
  if (!dOd || !dQd || !dKd || !dVd || !aligned(dOd, 16) || !aligned(dQd, 16) || !aligned(dKd, 16) ||
      !aligned(dVd, 16) || !workspace || !aligned(workspace, 16) ||
      workspace_bytes < osattn_bwd_workspace_bytes(B, H, Nq) || heads_per_chunk < 0)
    return OSATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  rc = device_state(&ds);
  if (rc != OSATTN_OK) return rc;
  // Each chunk's D goes where the whole call's D of its heads would; when
  // those places are 16-byte aligned (Nq a multiple of 4) the chunks'
  // kernels may alternate between two compute streams, otherwise they run
  // in order on `stream` and share the start of the workspace.  Two waves of
  // dK/dV CTAs a chunk (128 keys per CTA on the tensor cores, 32 in the fp32
  // kernels): from pinned host memory, B8 H40 2048 d128 5.48 ms a call and
  // causal B1 H32 16K d128 5.18 ms, against 5.93 / 5.05 with one wave and
  // 5.51 / 5.71 on one stream.
  const bool alternate = Nq % 4 == 0;
  const int hc = offload_heads(heads_per_chunk, H, Nkv, dtype == OSATTN_FP32 ? 32 : 128, ds->num_sms,
                               2);
  const size_t es = elem_size(dtype);
  const size_t qb = static_cast<size_t>(Nq) * d * es, kb = static_cast<size_t>(Nkv) * d * es;
  const size_t lb = static_cast<size_t>(Nq) * sizeof(float);
  const OffloadSeg ins[6] = {{const_cast<void*>(Qh), Qd, qb},   {const_cast<void*>(Kh), Kd, kb},
                             {const_cast<void*>(Vh), Vd, kb},   {const_cast<void*>(Oh), Od, qb},
                             {const_cast<void*>(dOh), dOd, qb}, {const_cast<float*>(LSEh), LSEd, lb}};
  const OffloadSeg outs[3] = {{dQh, dQd, qb}, {dKh, dKd, kb}, {dVh, dVd, kb}};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return offload_pipeline(ds, cs, B, H, hc, ins, 6, outs, 3, alternate, [&](int b, int h0, int nh,
                                                                cudaStream_t ks) {
    const size_t head0 = static_cast<size_t>(b) * H + h0;
    auto at = [&](const void* base, size_t head_bytes) {
      return static_cast<const char*>(base) + head0 * head_bytes;
    };
    auto at_w = [&](void* base, size_t head_bytes) {
      return static_cast<char*>(base) + head0 * head_bytes;
    };
    const size_t wo = alternate ? head0 * Nq * sizeof(float) : 0;
    return bwd_impl(at(Qd, qb), at(Kd, kb), at(Vd, kb), at(Od, qb), at(dOd, qb), LSEd + head0 * Nq,
                    at_w(dQd, qb), at_w(dKd, kb), at_w(dVd, kb), 1, nh, Nq, Nkv, d, nullptr, scale,
                    causal, key_len ? key_len + b : nullptr, dtype, static_cast<char*>(workspace) + wo,
                    workspace_bytes - wo, ks);
  });
}

int softmax_rows_offload_impl(const void* in_h, void* out_h, float* lse_h, void* in, void* out,
                              float* lse, int64_t rows, int N, int dtype, int64_t rows_per_chunk,
                              void* stream) {
  if (!in_h || !out_h || !in || !out || rows < 1 || N < 1 || rows_per_chunk < 0 ||
      (lse_h == nullptr) != (lse == nullptr) || rows > 0x7fffffffLL)
    return OSATTN_ERR_INVALID_ARG;
  if (dtype != OSATTN_BF16 && dtype != OSATTN_FP32 && dtype != OSATTN_FP16)
    return OSATTN_ERR_UNSUPPORTED;
  const uintptr_t el = elem_size(dtype);
  if (!aligned(in, el) || !aligned(out, el) || (lse && !aligned(lse, 4)))
    return OSATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != OSATTN_OK) return rc;
  // Automatic: 16 chunks (the kernel is bound by memory, so the pipeline only
  // has to keep both copy directions busy; more chunks shorten its fill).
  int64_t rc_rows = rows_per_chunk ? rows_per_chunk : (rows + 15) / 16;
  if (rc_rows > rows) rc_rows = rows;
  const size_t rb = static_cast<size_t>(N) * el;
  const OffloadSeg ins[1] = {{const_cast<void*>(in_h), in, rb}};
  const OffloadSeg outs[2] = {{out_h, out, rb}, {lse_h, lse, sizeof(float)}};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return offload_pipeline(ds, cs, 1, static_cast<int>(rows), static_cast<int>(rc_rows), ins, 1, outs,
                          lse ? 2 : 1, true, [&](int, int r0, int nr, cudaStream_t ks) {
                            const size_t off = static_cast<size_t>(r0) * rb;
                            const cudaError_t e = osattn::launch_softmax_rows(
                                static_cast<const char*>(in) + off, static_cast<char*>(out) + off,
                                lse ? lse + r0 : nullptr, nr, N, dtype, ds->num_sms,
                                ds->row_cluster_max, ks);
                            return e == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
                          });
}

}  // namespace

namespace osattn {

int validate_splitkv(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                     int B, int H, int Nq, int Nkv, int d, float scale, const int32_t* key_len,
                     int dtype, int num_splits) {
  const int rc = validate_fwd(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, key_len, dtype);
  if (rc != OSATTN_OK) return rc;
  if (dtype == OSATTN_FP32) return OSATTN_ERR_UNSUPPORTED;
  if (num_splits < 1 || num_splits > OSATTN_MAX_SPLITS) return OSATTN_ERR_INVALID_ARG;
  return OSATTN_OK;
}

}  // namespace osattn

extern "C" {

int osattn_softmax_rows_offload(const void* in_host, void* out_host, float* lse_host, void* in,
                                void* out, float* lse, int64_t rows, int N, int dtype,
                                int64_t rows_per_chunk, void* stream) {
  return softmax_rows_offload_impl(in_host, out_host, lse_host, in, out, lse, rows, N, dtype,
                                   rows_per_chunk, stream);
}

int osattn_fwd_offload(const void* Q_host, const void* K_host, const void* V_host, void* O_host,
                       float* LSE_host, void* Q, void* K, void* V, void* O, float* LSE, int B,
                       int H, int Nq, int Nkv, int d, float scale, int causal,
                       const int32_t* key_len, int dtype, int heads_per_chunk, void* stream) {
  return fwd_offload_impl(Q_host, K_host, V_host, O_host, LSE_host, Q, K, V, O, LSE, B, H, Nq, Nkv,
                          d, scale, causal, key_len, dtype, heads_per_chunk, stream);
}

int osattn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
               int Nq, int Nkv, int d, float scale, int causal, const int32_t* key_len,
               int dtype, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, Nq, Nkv, d, nullptr, nullptr, nullptr, nullptr, scale,
                  causal, key_len, dtype, stream);
}

int osattn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                       int H, int Nq, int Nkv, int d, const int64_t* q_strides,
                       const int64_t* k_strides, const int64_t* v_strides,
                       const int64_t* o_strides, float scale, int causal,
                       const int32_t* key_len, int dtype, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, Nq, Nkv, d, q_strides, k_strides, v_strides, o_strides,
                  scale, causal, key_len, dtype, stream);
}

size_t osattn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  return static_cast<size_t>(num_splits) * rows * (static_cast<size_t>(d) + 1) * sizeof(float);
}

int osattn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                       int H, int Nq, int Nkv, int d, float scale, int causal,
                       const int32_t* key_len, int dtype, int num_splits, void* workspace,
                       size_t workspace_bytes, void* stream) {
  int rc = osattn::validate_splitkv(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, key_len, dtype,
                                    num_splits);
  if (rc != OSATTN_OK) return rc;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < osattn_splitkv_workspace_bytes(B, H, Nq, d, num_splits))
    return OSATTN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != OSATTN_OK) return rc;
  osattn::FwdArgs a = make_args(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, causal, key_len, stream, st);
  a.fp16 = dtype == OSATTN_FP16;
  take_strides(nullptr, H, Nq, d, dtype, a.q_strides);
  take_strides(nullptr, H, Nkv, d, dtype, a.k_strides);
  take_strides(nullptr, H, Nkv, d, dtype, a.v_strides);
  take_strides(nullptr, H, Nq, d, dtype, a.o_strides);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = o_part + static_cast<size_t>(num_splits) * B * H * Nq * d;
  return launch_splitkv(a, num_splits, o_part, lse_part);
}

size_t osattn_bwd_workspace_bytes(int B, int H, int Nq) {
  if (B < 1 || H < 1 || Nq < 1) return 0;
  return static_cast<size_t>(B) * H * Nq * sizeof(float);
}

}  // extern "C"

namespace {

int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nkv, int d,
             const int64_t* const* strides, float scale, int causal, const int32_t* key_len,
             int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_fwd(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, key_len, dtype);
  if (rc != OSATTN_OK) return rc;
  if (!dO || !dQ || !dK || !dV || !aligned(dO, 16) || !aligned(dQ, 16) || !aligned(dK, 16) ||
      !aligned(dV, 16))
    return OSATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < osattn_bwd_workspace_bytes(B, H, Nq))
    return OSATTN_ERR_INVALID_ARG;
  // strides: Q, K, V, O, dO, dQ, dK, dV (null array or null entries: contiguous)
  long long st[8][3];
  const int rows_of[8] = {Nq, Nkv, Nkv, Nq, Nq, Nq, Nkv, Nkv};
  for (int i = 0; i < 8; ++i)
    if (take_strides(strides ? strides[i] : nullptr, H, rows_of[i], d, dtype, st[i]) != OSATTN_OK)
      return OSATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  rc = device_state(&ds);
  if (rc != OSATTN_OK) return rc;
  osattn::BwdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.dO = dO;
  a.LSE = LSE;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.D = static_cast<float*>(workspace);
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nkv = Nkv;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.key_len = key_len;
  a.fp16 = dtype == OSATTN_FP16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = ds->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.num_sms = ds->num_sms;
  long long* dst[8] = {a.q_strides, a.k_strides, a.v_strides, a.o_strides, a.do_strides,
                       a.dq_strides, a.dk_strides, a.dv_strides};
  for (int i = 0; i < 8; ++i)
    for (int j = 0; j < 3; ++j) dst[i][j] = st[i][j];
  if (dtype == OSATTN_FP32)
    return osattn::launch_bwd_fp32(a) == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
  CUtensorMap tmQ, tmK, tmV, tmdO;
  if (encode_map(&tmQ, Q, a.fp16, d, Nq, H, B, st[0]) != OSATTN_OK ||
      encode_map(&tmK, K, a.fp16, d, Nkv, H, B, st[1]) != OSATTN_OK ||
      encode_map(&tmV, V, a.fp16, d, Nkv, H, B, st[2]) != OSATTN_OK ||
      encode_map(&tmdO, dO, a.fp16, d, Nq, H, B, st[4]) != OSATTN_OK)
    return OSATTN_ERR_CUDA;
  return osattn::launch_bwd(a, tmQ, tmK, tmV, tmdO) == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int osattn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
               const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nkv,
               int d, float scale, int causal, const int32_t* key_len, int dtype,
               void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nkv, d, nullptr, scale, causal,
                  key_len, dtype, workspace, workspace_bytes, stream);
}

int osattn_bwd_offload(const void* Q_host, const void* K_host, const void* V_host,
                       const void* O_host, const void* dO_host, const float* LSE_host,
                       void* dQ_host, void* dK_host, void* dV_host, void* Q, void* K, void* V,
                       void* O, void* dO, float* LSE, void* dQ, void* dK, void* dV, int B, int H,
                       int Nq, int Nkv, int d, float scale, int causal, const int32_t* key_len,
                       int dtype, void* workspace, size_t workspace_bytes, int heads_per_chunk,
                       void* stream) {
  return bwd_offload_impl(Q_host, K_host, V_host, O_host, dO_host, LSE_host, dQ_host, dK_host,
                          dV_host, Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nkv, d, scale, causal,
                          key_len, dtype, workspace, workspace_bytes, heads_per_chunk, stream);
}

int osattn_bwd_strided(const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                       int H, int Nq, int Nkv, int d, const int64_t* q_strides,
                       const int64_t* k_strides, const int64_t* v_strides,
                       const int64_t* o_strides, const int64_t* do_strides,
                       const int64_t* dq_strides, const int64_t* dk_strides,
                       const int64_t* dv_strides, float scale, int causal,
                       const int32_t* key_len, int dtype, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const int64_t* st[8] = {q_strides, k_strides, v_strides, o_strides,
                          do_strides, dq_strides, dk_strides, dv_strides};
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nkv, d, st, scale, causal, key_len,
                  dtype, workspace, workspace_bytes, stream);
}

int osattn_softmax_rows(const void* in, void* out, float* lse, int64_t rows, int N, int dtype,
                        void* stream) {
  if (!in || !out || rows < 1 || N < 1) return OSATTN_ERR_INVALID_ARG;
  if (dtype != OSATTN_BF16 && dtype != OSATTN_FP32 && dtype != OSATTN_FP16)
    return OSATTN_ERR_UNSUPPORTED;
  const uintptr_t el = elem_size(dtype);
  if (!aligned(in, el) || !aligned(out, el) || (lse && !aligned(lse, 4)))
    return OSATTN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != OSATTN_OK) return rc;
  const cudaError_t e = osattn::launch_softmax_rows(in, out, lse, static_cast<long long>(rows), N,
                                                    dtype, st->num_sms, st->row_cluster_max,
                                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
}

int osattn_step_trace_read(void* host, size_t bytes, size_t* needed) {
  size_t n = 0;
  const cudaError_t e = osattn::read_step_trace(host, bytes, &n);
  if (needed) *needed = n;
  if (e == cudaErrorNotSupported) return OSATTN_ERR_UNSUPPORTED;
  if (e == cudaErrorInvalidValue) return OSATTN_ERR_INVALID_ARG;
  return e == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
}

int osattn_get_device_status(void* stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != OSATTN_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  unsigned int host[2] = {0, 0};
  if (cudaMemcpy(host, st->status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  const unsigned int zero[2] = {0, 0};
  if (cudaMemcpy(st->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return OSATTN_ERR_CUDA;
  if (host[0] != 0) g_last_timeout_site.store(static_cast<int>(host[1]));
  return host[0] == 0 ? OSATTN_OK : static_cast<int>(host[0]);
}

int osattn_last_timeout_site(void) { return g_last_timeout_site.load(); }

uint64_t osattn_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns < 1000 ? 1000 : ns);
}

int osattn_test_wait_timeout(void* stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != OSATTN_OK) return rc;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st->status,
                                                                      g_wait_limit_ns.load());
  return cudaGetLastError() == cudaSuccess ? OSATTN_OK : OSATTN_ERR_CUDA;
}

}  // extern "C"
