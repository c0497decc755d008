// The C ABI of include/tl.h: argument validation, the per-device status word
// and the kernel launches. Validation happens before any CUDA call, so argument
// errors return without touching the device (and work without a GPU).
#include "tl_internal.cuh"

#include <mutex>

namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

// Device address of this device's status word (resolved once per device).
int status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TL_ECUDA;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return TL_ECUDA;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return TL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_nk(int N, int K) {
  if (N < 0 || K <= 0) return TL_EINVAL;
  if (K % tl::kBlock != 0 || K > tl::kMaxK) return TL_EUNSUPPORTED;
  if (N % 128 != 0) return TL_EUNSUPPORTED;
  return TL_OK;
}

int check_linear(const void* packed, const void* qT, const void* sw, const void* xq,
                 const void* sx, int M, int N, int K, const void* y, int y_dtype,
                 const void* acc_dbg) {
  if (M < 0) return TL_EINVAL;
  int r = check_nk(N, K);
  if (r != TL_OK) return r;
  if (y_dtype != TL_BF16 && y_dtype != TL_F32) return TL_EINVAL;
  if (M == 0 || N == 0) return TL_OK;
  if (!packed || !qT || !sw || !xq || !sx || !y) return TL_EINVAL;
  if (!aligned16(packed) || !aligned16(qT) || !aligned16(sw) || !aligned16(xq) ||
      !aligned16(sx) || !aligned16(y) || (acc_dbg && !aligned16(acc_dbg)))
    return TL_EINVAL;
  return TL_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// A wait that nothing ends: phase 0 of a fresh mbarrier with no arrival. The
// bounded wait gives up after limit_ns and records TL_ETIMEOUT, the path every
// kernel of the library takes when one of its waits runs out.
__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tl::mbar_init(tl::smem_u32(&bar), 1);
    tl::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tl::mbar_wait(tl::smem_u32(&bar), 0, nullptr, limit_ns))
    tl::set_status(status, TL_ETIMEOUT);
}

}  // namespace

extern "C" {

const char* tl_strerror(int status) {
  switch (status) {
    case TL_OK: return "TL_OK";
    case TL_EINVAL: return "TL_EINVAL: invalid argument (NULL, negative size, misaligned, bad dtype)";
    case TL_EUNSUPPORTED: return "TL_EUNSUPPORTED: unsupported shape";
    case TL_ECUDA: return "TL_ECUDA: CUDA runtime or launch error";
    case TL_ETIMEOUT: return "TL_ETIMEOUT: a bounded device-side wait gave up";
    case TL_EDATA: return "TL_EDATA: input data out of range";
    case TL_ENOSPACE: return "TL_ENOSPACE: size exceeds the provided capacity";
    default: return "unknown tl_status";
  }
}

int tl_version(void) { return 10000; }

int tl_packed_sizes(int N, int K, size_t* packed_bytes, size_t* qT_bytes, size_t* sw_bytes) {
  const int r = check_nk(N, K);
  if (r != TL_OK) return r;
  if (packed_bytes) *packed_bytes = static_cast<size_t>(N) * K / 4;
  if (qT_bytes) *qT_bytes = static_cast<size_t>(K / tl::kGroup) * N;
  if (sw_bytes) *sw_bytes = static_cast<size_t>(N) * 4;
  return TL_OK;
}

int tl_pack_weights(const int8_t* codes, const uint16_t* s, int N, int K, uint8_t* packed,
                    int8_t* qT, float* sw, void* stream) {
  int r = check_nk(N, K);
  if (r != TL_OK) return r;
  if (N == 0) return TL_OK;
  if (!codes || !s || !packed || !qT || !sw) return TL_EINVAL;
  if (!aligned16(codes) || !aligned16(s) || !aligned16(packed) || !aligned16(qT) || !aligned16(sw))
    return TL_EINVAL;
  int* status = nullptr;
  if ((r = status_ptr(&status)) != TL_OK) return r;
  return tl::launch_pack(codes, s, N, K, reinterpret_cast<uint32_t*>(packed), qT, sw, status,
                         as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_rotate_quant_act(const uint16_t* x, int M, int K, const int8_t* signs, void* xq,
                        int xq_dtype, float* sx, void* stream) {
  if (M < 0 || K <= 0) return TL_EINVAL;
  if (K % tl::kBlock != 0 || K > tl::kMaxK) return TL_EUNSUPPORTED;
  if (xq_dtype != TL_I8 && xq_dtype != TL_F16) return TL_EINVAL;
  if (M == 0) return TL_OK;
  if (!x || !xq || !sx) return TL_EINVAL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(sx) || (signs && !aligned16(signs)))
    return TL_EINVAL;
  return tl::launch_rotate_quant(x, M, K, signs, xq, xq_dtype, sx, as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_prefill_workspace_size(int M, int N, int K, size_t* bytes) {
  if (bytes == nullptr || M < 0) return TL_EINVAL;
  const int r = check_nk(N, K);
  if (r != TL_OK) return r;
  *bytes = 0;
  if (M == 0 || N == 0) return TL_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TL_ECUDA;
  *bytes = tl::prefill_workspace_bytes(M, N, K, sms);
  return TL_OK;
}

int tl_linear_prefill(const uint8_t* packed, const int8_t* qT, const float* sw,
                      const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                      int y_dtype, int32_t* acc_dbg, void* workspace, size_t ws_bytes,
                      void* stream) {
  int r = check_linear(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg);
  if (r != TL_OK || M == 0 || N == 0) return r;
  if (workspace && !aligned16(workspace)) return TL_EINVAL;
  int* status = nullptr;
  if ((r = status_ptr(&status)) != TL_OK) return r;
  tl::PrefillArgs a{packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, workspace, ws_bytes, false};
  cudaError_t ce;
  return tl::launch_prefill(a, status, as_stream(stream), &ce);
}

int tl_linear_prefill_noalloc(const uint8_t* packed, const int8_t* qT, const float* sw,
                              const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                              int y_dtype, int32_t* acc_dbg, void* stream) {
  int r = check_linear(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg);
  if (r != TL_OK || M == 0 || N == 0) return r;
  size_t need = 0;
  if ((r = tl_prefill_workspace_size(M, N, K, &need)) != TL_OK) return r;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TL_ECUDA;
  // with fewer tiles than SMs the split is the point: refuse what does not fit;
  // with more, a split without room runs every tile whole
  if (need > tl::kNoAllocScratchBytes && tl::prefill_split_required(M, N, sms)) return TL_ENOSPACE;
  int* status = nullptr;
  if ((r = status_ptr(&status)) != TL_OK) return r;
  void* scratch = nullptr;
  if ((r = tl::prefill_noalloc_scratch(&scratch)) != TL_OK) return r;
  tl::PrefillArgs a{packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, scratch,
                    tl::kNoAllocScratchBytes, true};
  cudaError_t ce;
  return tl::launch_prefill(a, status, as_stream(stream), &ce);
}

int tl_linear_decode(const uint8_t* packed, const int8_t* qT, const float* sw, const int8_t* xq,
                     const float* sx, int M, int N, int K, void* y, int y_dtype,
                     int32_t* acc_dbg, void* stream) {
  int r = check_linear(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg);
  if (r != TL_OK) return r;
  if (M > tl::kMaxDecodeM) return TL_EUNSUPPORTED;
  if (M == 0 || N == 0) return TL_OK;
  return tl::launch_decode(reinterpret_cast<const uint32_t*>(packed), qT, sw, xq, sx, M, N, K, y,
                           y_dtype, acc_dbg, as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_linear_decode_tc(const uint8_t* packed, const int8_t* qT, const float* sw,
                        const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                        int y_dtype, int32_t* acc_dbg, void* stream) {
  int r = check_linear(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg);
  if (r != TL_OK) return r;
  if (M > tl::kMaxDecodeM) return TL_EUNSUPPORTED;
  if (M == 0 || N == 0) return TL_OK;
  int* status = nullptr;
  if ((r = status_ptr(&status)) != TL_OK) return r;
  return tl::launch_decode_tc(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, status,
                              as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_linear_decode_fused(const uint8_t* packed, const int8_t* qT, const float* sw,
                           const uint16_t* x, const int8_t* signs, int M, int N, int K, void* y,
                           int y_dtype, int32_t* acc_dbg, int8_t* xq_out, float* sx_out,
                           void* stream) {
  int r = check_linear(packed, qT, sw, x, sw, M, N, K, y, y_dtype, acc_dbg);
  if (r != TL_OK) return r;
  if (M > 16 || (M == 1 && K > tl::kMaxFusedDecodeK)) return TL_EUNSUPPORTED;
  if (M == 0 || N == 0) return TL_OK;
  if ((signs && !aligned16(signs)) || (xq_out && !aligned16(xq_out)) || (sx_out && !aligned16(sx_out)))
    return TL_EINVAL;
  if (M == 1)
    return tl::launch_decode_fused(reinterpret_cast<const uint32_t*>(packed), qT, sw, x, signs, N,
                                   K, y, y_dtype, acc_dbg, xq_out, sx_out,
                                   as_stream(stream)) == cudaSuccess
               ? TL_OK
               : TL_ECUDA;
  bool supported = false;
  const cudaError_t e = tl::launch_decode_fused_m(reinterpret_cast<const uint32_t*>(packed), qT, sw,
                                                  x, signs, M, N, K, y, y_dtype, acc_dbg, xq_out,
                                                  sx_out, as_stream(stream), &supported);
  if (!supported) return TL_EUNSUPPORTED;
  return e == cudaSuccess ? TL_OK : TL_ECUDA;
}

int tl_rotate_act(const uint16_t* x, int M, int K, const int8_t* signs, float* xr, void* stream) {
  if (M < 0 || K <= 0) return TL_EINVAL;
  if (K % tl::kBlock != 0 || K > tl::kMaxK) return TL_EUNSUPPORTED;
  if (M == 0) return TL_OK;
  if (!x || !xr) return TL_EINVAL;
  if (!aligned16(x) || !aligned16(xr) || (signs && !aligned16(signs))) return TL_EINVAL;
  return tl::launch_rotate(x, M, K, signs, xr, as_stream(stream)) == cudaSuccess ? TL_OK : TL_ECUDA;
}

int tl_linear_decode_f32act(const uint8_t* packed, const uint16_t* s, const float* xr, int M, int N,
                            int K, void* y, int y_dtype, void* stream) {
  if (M < 0) return TL_EINVAL;
  int r = check_nk(N, K);
  if (r != TL_OK) return r;
  if (y_dtype != TL_BF16 && y_dtype != TL_F32) return TL_EINVAL;
  if (M > tl::kMaxF32ActM || static_cast<long long>(M) * K > tl::kMaxF32ActMK) return TL_EUNSUPPORTED;
  if (M == 0 || N == 0) return TL_OK;
  if (!packed || !s || !xr || !y) return TL_EINVAL;
  if (!aligned16(packed) || !aligned16(s) || !aligned16(xr) || !aligned16(y)) return TL_EINVAL;
  return tl::launch_decode_f32act(packed, s, xr, M, N, K, y, y_dtype, as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_codec_quant(const uint16_t* x, int R, int H, int8_t* q, float* scale, void* stream) {
  if (R < 0 || H <= 0) return TL_EINVAL;
  if (H % tl::kGroup != 0) return TL_EUNSUPPORTED;
  if (R == 0) return TL_OK;
  if (!x || !q || !scale) return TL_EINVAL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return TL_EINVAL;
  return tl::launch_codec_quant(x, R, H, q, scale, as_stream(stream)) == cudaSuccess ? TL_OK
                                                                                      : TL_ECUDA;
}

int tl_codec_dequant_add(const uint16_t* own, const int8_t* q_peers, const float* scale_peers,
                         int npeers, int R, int H, uint16_t* out, void* stream) {
  if (R < 0 || H <= 0 || npeers < 0) return TL_EINVAL;
  if (H % tl::kGroup != 0 || npeers > tl::kMaxCodecPeers) return TL_EUNSUPPORTED;
  if (R == 0) return TL_OK;
  if (!own || !out || (npeers > 0 && (!q_peers || !scale_peers))) return TL_EINVAL;
  if (!aligned16(own) || !aligned16(out) || (npeers > 0 && (!aligned16(q_peers) || !aligned16(scale_peers))))
    return TL_EINVAL;
  return tl::launch_codec_dequant_add(own, q_peers, scale_peers, npeers, R, H, out,
                                      as_stream(stream)) == cudaSuccess
             ? TL_OK
             : TL_ECUDA;
}

int tl_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 100000) return TL_EINVAL;
  int* status = nullptr;
  const int r = status_ptr(&status);
  if (r != TL_OK) return r;
  wait_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>(status, 1000ull * limit_us);
  return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ECUDA;
}

int tl_get_status(void* stream) {
  int* status = nullptr;
  int r = status_ptr(&status);
  if (r != TL_OK) return r;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TL_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TL_ECUDA;
  const int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return TL_ECUDA;
  return v;
}

}  // extern "C"
