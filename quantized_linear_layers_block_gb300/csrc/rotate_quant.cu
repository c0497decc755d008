// K1: input-side block Hadamard rotation fused with per-token int8 quantisation.
//
// Qiita item ecc183fae033565af7cb: 前提 (a block-wise Hadamard rotation on the
// layer's input side), §1 "TP=2 への移植" (Sylvester structure, the last
// butterfly stage combines the two 512-halves) and §4 "効いた高速化"
// (activations quantised to int8 per token after the rotation).
//
// One CTA per token, one warp per 1024-column block (rotate_block_warp in
// tl_internal.cuh: the butterfly stages run in the order 1, 2, 4, ..., 512, so
// every element sees the same fp32 additions as a plain sequential FWHT).
#include "tl_internal.cuh"

#include <cuda_fp16.h>

namespace tl {
namespace {

template <int XQ_DTYPE>
__global__ void __launch_bounds__(1024)
rotate_quant_kernel(const uint16_t* __restrict__ x, int K, const int8_t* __restrict__ signs,
                    void* __restrict__ xq, float* __restrict__ sx) {
  __shared__ float warp_max[32];
  const int lane = threadIdx.x & 31;
  const int blk = threadIdx.x >> 5;
  const int nblk = blockDim.x >> 5;
  const size_t m = blockIdx.x;
  const size_t base = m * static_cast<size_t>(K) + static_cast<size_t>(blk) * kBlock;
  // x may be the output of the preceding kernel; once it is complete, the next
  // kernel (the layer's GEMM) may start its weight-only prologue.
  pdl_wait_prior();
  pdl_launch_dependents();

  float v[4][8];
  float amax = rotate_block_warp(x + base, signs == nullptr ? nullptr : signs + blk * kBlock, lane, v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) warp_max[blk] = amax;
  __syncthreads();
  float a = 0.f;
  for (int b = 0; b < nblk; ++b) a = fmaxf(a, warp_max[b]);

  const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
  if (threadIdx.x == 0) sx[m] = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;

#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      q[e] = quant_i8(v[j][e], inv);
    }
    const size_t off = base + 256 * j + 8 * lane;
    if (XQ_DTYPE == TL_I8) {
      uint2 o;
      o.x = (q[0] & 0xFF) | ((q[1] & 0xFF) << 8) | ((q[2] & 0xFF) << 16) | ((q[3] & 0xFF) << 24);
      o.y = (q[4] & 0xFF) | ((q[5] & 0xFF) << 8) | ((q[6] & 0xFF) << 16) | ((q[7] & 0xFF) << 24);
      *reinterpret_cast<uint2*>(static_cast<int8_t*>(xq) + off) = o;
    } else {
      uint32_t hw[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t lo = __half_as_ushort(__int2half_rn(q[2 * p]));
        const uint32_t hi = __half_as_ushort(__int2half_rn(q[2 * p + 1]));
        hw[p] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(xq) + off) =
          make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
  }
}

// The rotation alone, fp32 out (the float-activation decode's input).
__global__ void __launch_bounds__(1024)
rotate_kernel(const uint16_t* __restrict__ x, int K, const int8_t* __restrict__ signs,
              float* __restrict__ xr) {
  const int lane = threadIdx.x & 31;
  const int blk = threadIdx.x >> 5;
  const size_t base = blockIdx.x * static_cast<size_t>(K) + static_cast<size_t>(blk) * kBlock;
  pdl_wait_prior();
  pdl_launch_dependents();
  float v[4][8];
  rotate_block_warp(x + base, signs == nullptr ? nullptr : signs + blk * kBlock, lane, v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float4* o = reinterpret_cast<float4*>(xr + base + 256 * j + 8 * lane);
    o[0] = make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
    o[1] = make_float4(v[j][4], v[j][5], v[j][6], v[j][7]);
  }
}

}  // namespace

cudaError_t launch_rotate(const uint16_t* x, int M, int K, const int8_t* signs, float* xr,
                          cudaStream_t st) {
  return launch_pdl(rotate_kernel, dim3(M), dim3((K / kBlock) * 32), 0, st, x, K, signs, xr);
}

cudaError_t launch_rotate_quant(const uint16_t* x, int M, int K, const int8_t* signs, void* xq,
                                int xq_dtype, float* sx, cudaStream_t st) {
  const int threads = (K / kBlock) * 32;
  if (xq_dtype == TL_I8)
    return launch_pdl(rotate_quant_kernel<TL_I8>, dim3(M), dim3(threads), 0, st, x, K, signs, xq, sx);
  return launch_pdl(rotate_quant_kernel<TL_F16>, dim3(M), dim3(threads), 0, st, x, K, signs, xq, sx);
}

}  // namespace tl
