// K2f: decode (M <= 4) with floating-point activations.
//
// Qiita item ecc183fae033565af7cb §5 "効かなかったもの": the production decode
// keeps the activations in floating point and was more exact than the int8
// dp4a GEMV. This kernel computes that variant for the same packed weights:
//   y[m,n] = sum_g s[n,g] sum_{k in g} code[n,k] xr[m,k]
// with xr the fp32 rotation (tl_rotate_act), s the original fp16 group scales
// and fp32 arithmetic throughout; no activation quantisation, no int8 q.
//
// Layout and streaming follow the int8 decode kernel: 32 rows per CTA, 4 per
// warp; lane l owns the 32-code chunks l, l+32, ... of the rows (a warp reads
// 256 contiguous bytes of a row per step) and a ring of kRing chunk steps of
// the warp's four rows (codes and scales) runs ahead of the arithmetic, its
// first entries issued before the wait on the preceding kernel. A lane reads
// each staged activation chunk once and applies it to all four rows: the
// fp32 activations cost four bytes of shared-memory bandwidth per code, which
// bound the kernel when every row re-read them.
//
// Codes to floats without conversions: the 2-bit field e at bit 2j of a half
// word, or-ed into the mantissa of 1.5 * 2^23 (whose last mantissa bit is
// worth 1), gives the float 1.5 * 2^23 + e * 4^j; subtracting 1.5 * 2^23 + 4^j
// leaves (e - 1) * 4^j = code * 4^j exactly (all integers below 2^24). The activations are staged pre-scaled by
// 4^-j (j = (k mod 16) / 2, a power of two: exact for |xr| >= 2^-112), so each
// fused multiply-add adds code * xr exactly before its one rounding. The low
// and high half words hold the even and odd codes of the same j, so one
// packed fp32x2 add and one packed fp32x2 FMA per token handle two codes.
// Each field is placed by one LOP3 with its mask as the immediate and the
// magic in a register (with both as constants the compiler added a move per
// LOP3: 12.4 M -> 9.7 M instructions, 17.4 -> 14.9 us at M = 1).
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tl {
namespace {

constexpr int kFWarps = 8;
constexpr int kFRowsPerCta = 32;
constexpr int kRing = 2;          // chunk steps (4 rows each) of weights in flight
constexpr int kXStride = 36;   // floats per staged 32-code chunk: 4 pad, conflict-free float4 reads

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t f2_bits(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
// (x & (3 << 2 J)) | magic as one LOP3 with the mask as its immediate and the
// magic in a register
template <int J>
__device__ __forceinline__ uint32_t field_or(uint32_t x, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(3u << (2 * J)), "r"(magic));
  return d;
}
__device__ __forceinline__ uint32_t field_or_j(int j, uint32_t x, uint32_t magic) {
  switch (j) {
    case 0: return field_or<0>(x, magic);
    case 1: return field_or<1>(x, magic);
    case 2: return field_or<2>(x, magic);
    case 3: return field_or<3>(x, magic);
    case 4: return field_or<4>(x, magic);
    case 5: return field_or<5>(x, magic);
    case 6: return field_or<6>(x, magic);
    default: return field_or<7>(x, magic);
  }
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ void store_out(void* y, int y_dtype, size_t idx, float v) {
  if (y_dtype == TL_F32)
    static_cast<float*>(y)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

template <int MT>
__global__ void __launch_bounds__(kFWarps * 32)
decode_f32_kernel(const uint2* __restrict__ packed, const __half* __restrict__ s,
                  const float* __restrict__ xr, int M, int N, int K, void* __restrict__ y,
                  int y_dtype) {
  extern __shared__ __align__(16) float xs[];   // [MT][K/32][kXStride], pre-scaled by 4^-j
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int NC = K / 32;                        // chunks per row
  const int G = K / kGroup;
  const int PL = NC / 32;                       // chunk steps per lane
  const int n0 = blockIdx.x * kFRowsPerCta;
  // the warp's rows are n0 + warp + 8 r, r = 0..3
  const uint2* pw = packed + static_cast<size_t>(n0 + warp) * NC + lane;
  const __half* ps = s + static_cast<size_t>(n0 + warp) * G + (lane >> 2);
  const size_t wrow = static_cast<size_t>(kFWarps) * NC;   // uint2 between the warp's rows
  const size_t srow = static_cast<size_t>(kFWarps) * G;

  uint2 ring_w[kRing][4];
  __half ring_s[kRing][4];
#pragma unroll
  for (int u = 0; u < kRing; ++u) {
    if (u < PL) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        ring_w[u][r] = __ldg(pw + r * wrow + u * 32);
        ring_s[u][r] = ps[r * srow + u * 8];
      }
    }
  }
  pdl_launch_dependents();
  pdl_wait_prior();
  for (int i = tid; i < MT * (K / 4); i += blockDim.x) {
    const int m = i / (K / 4), k = 4 * (i - m * (K / 4));
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m < M) v = reinterpret_cast<const float4*>(xr + static_cast<size_t>(m) * K)[k / 4];
    const int j = (k & 15) >> 1;                                   // k, k+1 share j; k+2, k+3 have j+1
    const float s0 = __uint_as_float(static_cast<uint32_t>(127 - 2 * j) << 23);        // 4^-j
    const float s1 = __uint_as_float(static_cast<uint32_t>(127 - 2 * (j + 1)) << 23);  // 4^-(j+1)
    v.x = __fmul_rn(v.x, s0);
    v.y = __fmul_rn(v.y, s0);
    v.z = __fmul_rn(v.z, s1);
    v.w = __fmul_rn(v.w, s1);
    *reinterpret_cast<float4*>(xs + (static_cast<size_t>(m) * NC + k / 32) * kXStride + (k & 31)) = v;
  }
  __syncthreads();

  uint32_t magic_r;   // 1.5 * 2^23 (ulp 1), kept in a register for the LOP3s
  asm volatile("mov.b32 %0, 0x4B400000;" : "=r"(magic_r));
  float acc[4][MT];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

  for (int i0 = 0; i0 < PL; i0 += kRing) {
#pragma unroll
    for (int u = 0; u < kRing; ++u) {
      const int i = i0 + u;
      if (i < PL) {
        uint2 w[4];
        float sg[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          w[r] = ring_w[u][r];
          sg[r] = __half2float(ring_s[u][r]);
          if (i + kRing < PL) {
            ring_w[u][r] = __ldg(pw + r * wrow + (i + kRing) * 32);
            ring_s[u][r] = ps[r * srow + (i + kRing) * 8];
          }
        }
        const int c = i * 32 + lane;
        uint64_t t[4][MT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m) t[r][m] = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            lo[r] = q == 0 ? w[r].x : w[r].y;
            hi[r] = lo[r] >> 16;
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float4 x4[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m)
              x4[m] = *reinterpret_cast<const float4*>(
                  xs + (static_cast<size_t>(m) * NC + c) * kXStride + 16 * q + 4 * v);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int j = 2 * v + h;
              const float neg = -(12582912.0f + static_cast<float>(1u << (2 * j)));   // -(1.5 * 2^23 + 4^j)
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                uint64_t f = f2_bits(field_or_j(j, lo[r], magic_r), field_or_j(j, hi[r], magic_r));
                f = f2_add(f, f2(neg, neg));                                      // (even, odd) code * 4^j
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                  const uint64_t x2 = h == 0 ? f2(x4[m].x, x4[m].y) : f2(x4[m].z, x4[m].w);
                  t[r][m] = f2_fma(f, x2, t[r][m]);
                }
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            acc[r][m] = fmaf(sg[r], __fadd_rn(f2_lo(t[r][m]), f2_hi(t[r][m])), acc[r][m]);
      }
    }
  }
  // reduce the four rows together: lanes with bit 4 clear keep rows 0, 1, with it
  // set rows 2, 3; bit 3 then picks one; lanes 0, 8, 16, 24 end with rows 0..3
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const float s0 = (b4 ? acc[2][m] : acc[0][m]) + __shfl_xor_sync(0xffffffffu, b4 ? acc[0][m] : acc[2][m], 16);
    const float s1 = (b4 ? acc[3][m] : acc[1][m]) + __shfl_xor_sync(0xffffffffu, b4 ? acc[1][m] : acc[3][m], 16);
    float v = (b3 ? s1 : s0) + __shfl_xor_sync(0xffffffffu, b3 ? s0 : s1, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    if ((lane & 7) == 0 && m < M) {
      const int r = 2 * (lane >> 4) + ((lane >> 3) & 1);
      store_out(y, y_dtype, static_cast<size_t>(m) * N + n0 + warp + kFWarps * r, v);
    }
  }
}

template <int MT>
cudaError_t launch_f(const uint8_t* packed, const uint16_t* s, const float* xr, int M, int N, int K,
                     void* y, int y_dtype, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(MT) * (K / 32) * kXStride * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(decode_f32_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_f32_kernel<MT>, dim3(N / kFRowsPerCta), dim3(kFWarps * 32), smem, st,
                    reinterpret_cast<const uint2*>(packed), reinterpret_cast<const __half*>(s), xr, M,
                    N, K, y, y_dtype);
}

}  // namespace

cudaError_t launch_decode_f32act(const uint8_t* packed, const uint16_t* s, const float* xr, int M,
                                 int N, int K, void* y, int y_dtype, cudaStream_t st) {
  if (M <= 1) return launch_f<1>(packed, s, xr, M, N, K, y, y_dtype, st);
  // two tokens per launch: the weights of a 2-token pass are re-read from L2
  const size_t ysz = y_dtype == TL_F32 ? 4 : 2;
  for (int m0 = 0; m0 < M; m0 += 2) {
    const int mt = M - m0 < 2 ? M - m0 : 2;
    void* ym = static_cast<uint8_t*>(y) + static_cast<size_t>(m0) * N * ysz;
    const cudaError_t e = mt == 1
        ? launch_f<1>(packed, s, xr + static_cast<size_t>(m0) * K, 1, N, K, ym, y_dtype, st)
        : launch_f<2>(packed, s, xr + static_cast<size_t>(m0) * K, 2, N, K, ym, y_dtype, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace tl
