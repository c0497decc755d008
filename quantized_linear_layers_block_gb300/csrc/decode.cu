// K2: decode-time (M <= 32) ternary linear layer on the CUDA cores.
//
// Same integer accumulator and epilogue as the prefill GEMM of Qiita item
// ecc183fae033565af7cb §4 "効いた高速化"; the int8-activation GEMV with dp4a
// is the idea of §5 "効かなかったもの" (a dp4a decode GEMV), here computing
// exactly the quantised layer so that decode and prefill agree bit for bit.
//
// Each CTA owns 32 consecutive output rows. The activations of all tokens
// for a slab of K are staged in shared memory once, permuted so that a
// 32-bit word of packed codes shifted by 2t and masked with 0x03030303 lines
// up byte for byte with activation word t:
//   e-bytes of (w >> 2t) & 0x03030303  ->  k = 2t, 2t+8, 2t+1, 2t+9
// dp4a(e, x) then gives sum (code + 1) x; the per-chunk activation sum is
// subtracted and the result multiplied by q[n, g] (integer, exact).
// Lane l of a warp always owns the 32-code chunks l, l+32, ... of a row, so
// a warp-wide load of one row is fully coalesced 8-byte accesses.
#include "tl_internal.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace {

constexpr int kDecWarps = 8;
constexpr int kRowsPerCta = 32;
constexpr int kQStride = kRowsPerCta + 4;   // padded: conflict-free q reads
constexpr int kLoadBatch = 8;               // chunk loads in flight per lane
constexpr size_t kSlabBudget = 96 * 1024;

__host__ __device__ constexpr int slab_k(int mt, int K) {
  // bytes per slab column: mt activations + mt/8 chunk sums (4 bytes per 32 codes)
  const size_t per_k = static_cast<size_t>(mt) * 9 / 8;
  size_t ks = kSlabBudget / per_k;
  ks = ks / kBlock * kBlock;
  if (ks < kBlock) ks = kBlock;
  return static_cast<int>(ks < static_cast<size_t>(K) ? ks : K);
}

__device__ __forceinline__ void store_y(void* y, int y_dtype, size_t idx, float v) {
  if (y_dtype == TL_F32)
    static_cast<float*>(y)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

template <int MT>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
              const float* __restrict__ sw, const int8_t* __restrict__ xq,
              const float* __restrict__ sx, int M, int N, int K, int KS, void* __restrict__ y,
              int y_dtype, int32_t* __restrict__ acc_dbg) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = K / kGroup;
  uint32_t* xw = reinterpret_cast<uint32_t*>(smem);                         // [MT][KS/4]
  int32_t* csum = reinterpret_cast<int32_t*>(smem + static_cast<size_t>(MT) * KS);  // [MT][KS/32]
  int8_t* qs = reinterpret_cast<int8_t*>(smem + static_cast<size_t>(MT) * KS * 9 / 8);  // [G][kQStride]
  int32_t* part = reinterpret_cast<int32_t*>(
      smem + static_cast<size_t>(MT) * KS * 9 / 8 + ((static_cast<size_t>(G) * kQStride + 15) & ~size_t(15)));  // [32][MT]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n0 = blockIdx.x * kRowsPerCta;

  // q of this CTA's rows, all groups (qT is group-major: 32 contiguous bytes per group).
  for (int i = tid; i < G * (kRowsPerCta / 4); i += blockDim.x) {
    const int g = i / (kRowsPerCta / 4), r4 = i % (kRowsPerCta / 4);
    const uint32_t v =
        *reinterpret_cast<const uint32_t*>(qT + static_cast<size_t>(g) * N + n0 + 4 * r4);
    *reinterpret_cast<uint32_t*>(qs + g * kQStride + 4 * r4) = v;
  }

  const int nslab = (K + KS - 1) / KS;
  for (int sl = 0; sl < nslab; ++sl) {
    const int k0 = sl * KS;
    const int ks = min(KS, K - k0);
    const int nchunk = ks / 32;
    __syncthreads();  // previous slab fully consumed
    // Stage activations: one 32-code chunk per thread iteration.
    for (int i = tid; i < MT * nchunk; i += blockDim.x) {
      const int m = i / nchunk, c = i % nchunk;
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (m < M) {
        const uint4* src =
            reinterpret_cast<const uint4*>(xq + static_cast<size_t>(m) * K + k0 + 32 * c);
        u0 = src[0];
        u1 = src[1];
      }
      uint4 p0, p1;
      p0.x = __byte_perm(u0.x, u0.z, 0x5140);
      p0.y = __byte_perm(u0.x, u0.z, 0x7362);
      p0.z = __byte_perm(u0.y, u0.w, 0x5140);
      p0.w = __byte_perm(u0.y, u0.w, 0x7362);
      p1.x = __byte_perm(u1.x, u1.z, 0x5140);
      p1.y = __byte_perm(u1.x, u1.z, 0x7362);
      p1.z = __byte_perm(u1.y, u1.w, 0x5140);
      p1.w = __byte_perm(u1.y, u1.w, 0x7362);
      uint4* dst = reinterpret_cast<uint4*>(xw + static_cast<size_t>(m) * (KS / 4) + 8 * c);
      dst[0] = p0;
      dst[1] = p1;
      int s = 0;
      s = __dp4a(static_cast<int>(u0.x), 0x01010101, s);
      s = __dp4a(static_cast<int>(u0.y), 0x01010101, s);
      s = __dp4a(static_cast<int>(u0.z), 0x01010101, s);
      s = __dp4a(static_cast<int>(u0.w), 0x01010101, s);
      s = __dp4a(static_cast<int>(u1.x), 0x01010101, s);
      s = __dp4a(static_cast<int>(u1.y), 0x01010101, s);
      s = __dp4a(static_cast<int>(u1.z), 0x01010101, s);
      s = __dp4a(static_cast<int>(u1.w), 0x01010101, s);
      csum[m * (KS / 32) + c] = s;
    }
    __syncthreads();

    const int per_lane = nchunk / 32;  // ks is a multiple of 1024
    for (int r = warp; r < kRowsPerCta; r += kDecWarps) {
      const int n = n0 + r;
      const uint2* prow = reinterpret_cast<const uint2*>(packed + static_cast<size_t>(n) * (K / 16)) + k0 / 32;
      int acc[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = 0;

      for (int cb = 0; cb < per_lane; cb += kLoadBatch) {
        uint2 wv[kLoadBatch];
#pragma unroll
        for (int b = 0; b < kLoadBatch; ++b) {
          if (cb + b < per_lane) wv[b] = __ldg(prow + (cb + b) * 32 + lane);
        }
#pragma unroll
        for (int b = 0; b < kLoadBatch; ++b) {
          if (cb + b < per_lane) {
            const int c = (cb + b) * 32 + lane;          // chunk index within the slab
            const int g = (k0 + 32 * c) / kGroup;
            const int q = qs[g * kQStride + r];
            const int hsel = (c >> 2) & 1;                 // alternate halves: no bank conflicts
            const uint32_t wa = hsel ? wv[b].y : wv[b].x;
            const uint32_t wb = hsel ? wv[b].x : wv[b].y;
            int ea[4], eb[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              ea[t] = static_cast<int>((wa >> (2 * t)) & 0x03030303u);
              eb[t] = static_cast<int>((wb >> (2 * t)) & 0x03030303u);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint32_t* xm = xw + static_cast<size_t>(m) * (KS / 4) + 8 * c;
              const uint4 xa = *reinterpret_cast<const uint4*>(xm + 4 * hsel);
              const uint4 xb = *reinterpret_cast<const uint4*>(xm + 4 * (hsel ^ 1));
              int t = -csum[m * (KS / 32) + c];
              t = __dp4a(ea[0], static_cast<int>(xa.x), t);
              t = __dp4a(ea[1], static_cast<int>(xa.y), t);
              t = __dp4a(ea[2], static_cast<int>(xa.z), t);
              t = __dp4a(ea[3], static_cast<int>(xa.w), t);
              t = __dp4a(eb[0], static_cast<int>(xb.x), t);
              t = __dp4a(eb[1], static_cast<int>(xb.y), t);
              t = __dp4a(eb[2], static_cast<int>(xb.z), t);
              t = __dp4a(eb[3], static_cast<int>(xb.w), t);
              acc[m] += q * t;
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
      }
      // every lane now holds all MT totals; lane m owns token m
      int mine = 0;
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (lane == m) mine = acc[m];
      if (lane < MT) {
        if (sl > 0) mine += part[r * MT + lane];
        if (sl + 1 < nslab) {
          part[r * MT + lane] = mine;
        } else if (lane < M) {
          const size_t idx = static_cast<size_t>(lane) * N + n;
          if (acc_dbg != nullptr) acc_dbg[idx] = mine;
          const float v = __fmul_rn(__fmul_rn(__int2float_rn(mine), sw[n]), sx[lane]);
          store_y(y, y_dtype, idx, v);
        }
      }
    }
  }
}

template <int MT>
cudaError_t launch_mt(const uint32_t* packed, const int8_t* qT, const float* sw, const int8_t* xq,
                      const float* sx, int M, int N, int K, void* y, int y_dtype,
                      int32_t* acc_dbg, cudaStream_t st) {
  const int KS = slab_k(MT, K);
  const int G = K / kGroup;
  const size_t smem = static_cast<size_t>(MT) * KS * 9 / 8 +
                      ((static_cast<size_t>(G) * kQStride + 15) & ~size_t(15)) +
                      static_cast<size_t>(kRowsPerCta) * MT * 4;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int blocks = N / kRowsPerCta;
  decode_kernel<MT><<<blocks, kDecWarps * 32, smem, st>>>(packed, qT, sw, xq, sx, M, N, K, KS, y,
                                                          y_dtype, acc_dbg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const uint32_t* packed, const int8_t* qT, const float* sw,
                          const int8_t* xq, const float* sx, int M, int N, int K, void* y,
                          int y_dtype, int32_t* acc_dbg, cudaStream_t st) {
  if (M <= 1) return launch_mt<1>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 2) return launch_mt<2>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 4) return launch_mt<4>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 8) return launch_mt<8>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 16) return launch_mt<16>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  return launch_mt<32>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
}

}  // namespace tl
