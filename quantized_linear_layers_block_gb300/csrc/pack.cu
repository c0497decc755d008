// K0: load-time weight packing.
//
// Row-scale decomposition of Qiita item ecc183fae033565af7cb §4 "効いた高速化":
// the fp16 group scales s[n,g] become a per-row maximum smax[n] times an int8
// ratio q[n,g] = round(127 s[n,g] / smax[n]), so that code * q fits in int8.
// The 2-bit code storage of 前提 ("{-1,0,+1} の 2bit 表現") uses this
// library's own layout (documented in include/tl.h): the field at bit
// 16h + 2j of word w holds code[16w + 2j + h] + 1.
#include "tl_internal.cuh"

#include <cuda_fp16.h>

namespace tl {
namespace {

constexpr int kPackWarps = 8;

// One warp per row: smax, sw and q (written transposed), then the code words.
__global__ void __launch_bounds__(kPackWarps * 32)
pack_kernel(const int8_t* __restrict__ codes, const uint16_t* __restrict__ s, int N, int K,
            uint32_t* __restrict__ packed, int8_t* __restrict__ qT, float* __restrict__ sw,
            int* status) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * kPackWarps + (threadIdx.x >> 5);
  if (n >= N) return;
  const int G = K / kGroup;
  const uint16_t* srow = s + static_cast<size_t>(n) * G;

  float smax = 0.f;
  for (int g = lane; g < G; g += 32) {
    const float v = fabsf(__half2float(__ushort_as_half(srow[g])));
    smax = fmaxf(smax, v);
  }
  for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));

  for (int g = lane; g < G; g += 32) {
    int q = 0;
    if (smax > 0.f) {
      const float v = __half2float(__ushort_as_half(srow[g]));
      q = __float2int_rn(__fdiv_rn(__fmul_rn(127.f, v), smax));
    }
    qT[static_cast<size_t>(g) * N + n] = static_cast<int8_t>(q);
  }
  if (lane == 0) sw[n] = smax > 0.f ? __fdiv_rn(smax, 127.f) : 0.f;

  // 16 codes (16 bytes) per output word.
  const int W = K / 16;
  const uint4* crow = reinterpret_cast<const uint4*>(codes + static_cast<size_t>(n) * K);
  uint32_t* prow = packed + static_cast<size_t>(n) * W;
  bool bad = false;
  for (int w = lane; w < W; w += 32) {
    const uint4 c = crow[w];
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const int code = static_cast<int8_t>((cw[b >> 2] >> (8 * (b & 3))) & 0xFFu);
      bad |= (code < -1) | (code > 1);
      const uint32_t e = static_cast<uint32_t>(code + 1) & 3u;
      const int j = b >> 1, h = b & 1;
      word |= e << (16 * h + 2 * j);
    }
    prow[w] = word;
  }
  if (bad) set_status(status, TL_EDATA);
}

// Launched without programmatic serialization right after the pack kernel, so
// it starts only once the packed weights are complete and visible. The
// library's GEMM kernels read weights before they wait on the preceding kernel
// in the stream; with this launch in between, that preceding kernel is not
// the one that wrote the weights.
__global__ void pack_done_kernel() {}

}  // namespace

cudaError_t launch_pack(const int8_t* codes, const uint16_t* s, int N, int K, uint32_t* packed,
                        int8_t* qT, float* sw, int* status, cudaStream_t st) {
  const int blocks = (N + kPackWarps - 1) / kPackWarps;
  pack_kernel<<<blocks, kPackWarps * 32, 0, st>>>(codes, s, N, K, packed, qT, sw, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_done_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

}  // namespace tl
