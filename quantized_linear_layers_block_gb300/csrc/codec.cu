// int8 128-group codec of a row-parallel all-reduce payload, on one GPU.
//
// Qiita item ecc183fae033565af7cb §6 "最後に残った問題" (paragraph
// "通信を減らす・隠す、は全部だめだった"): each rank compresses its bf16 part
// to int8 with one scale per 128 elements, the parts are all-gathered, and
// each rank adds its own part, uncompressed, to the decompressed parts of the
// others. Item 66e136acefd5a54b2f1d §5 "解説: 長文を読む速度(prefill)" makes
// "compress" and "decompress and add" one GPU kernel each. The all-gather
// between them is the caller's.
//
// Both kernels stream: every byte is read once and written once, so they are
// bound by HBM bandwidth. Each CTA takes one batch of kCodecThreads * U
// vectors, so every load of the payload is issued as soon as its CTA starts
// (a loop of resident CTAs keeps fewer bytes in flight and measured slower).
// A thread owns 8 consecutive elements (one 16-byte bf16 vector) per step
// with U independent vectors in flight; 16 consecutive lanes cover one
// 128-element group, so the group maximum is four xor-shuffles within the
// half-warp. The quantiser is the layer's own:
// inv = fl32(127 / a), q = clamp(rne(fl32(x inv)), -127, 127), scale =
// fl32(a / 127); decompression is fl32(q scale) added in fp32 from the own
// part in peer order, rounded once to bf16. The two IEEE quotients of a group
// are computed once per warp lane (one lane per quotient), not by all 16 lanes
// of the group: 6.8 -> 6.3 us at 1584 x 5120.
#include "tl_internal.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace {

constexpr int kCodecThreads = 256;
constexpr int kQuantUnroll = 2;     // vectors per thread (compress)
constexpr int kDqUnroll = 4;        // vectors per thread (decompress and add)
constexpr int kVecPerGroup = kGroup / 8;   // 16 lanes per 128-element group

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}

// clamp(rne(v), -127, 127) as one byte, with NaN -> 0 (the value an fp32 ->
// int conversion gives it): the NaN-propagating max keeps a NaN a NaN, and the
// saturating conversion turns it into 0 and +inf into 127.
__device__ __forceinline__ uint32_t code_byte(float v) {
  float c;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(c) : "f"(v), "f"(-127.f));
  uint32_t r;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(r) : "f"(c));
  return r;
}

// Each thread quantises U vectors of 8 elements; the 2U groups of a warp need
// 4U IEEE quotients (127 / a and a / 127 per group), one per lane, exchanged by
// shuffles, instead of 2U per lane.
template <int U>
__global__ void __launch_bounds__(kCodecThreads)
codec_quant_kernel(const uint4* __restrict__ x, size_t nvec, uint2* __restrict__ q,
                   float* __restrict__ scale) {
  static_assert(4 * U <= 32, "one quotient per lane");
  pdl_wait_prior();   // x is normally the preceding kernel's output
  const int lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(blockIdx.x) * kCodecThreads * U + threadIdx.x;
  uint4 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const size_t idx = base + static_cast<size_t>(u) * kCodecThreads;
    v[u] = idx < nvec ? __ldcs(x + idx) : make_uint4(0, 0, 0, 0);
  }
  pdl_launch_dependents();
  float f[U][8], a[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    bf16x8_to_f32(v[u], f[u]);
    a[u] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) a[u] = fmaxf(a[u], fabsf(f[u][e]));
#pragma unroll
    for (int o = kVecPerGroup / 2; o > 0; o >>= 1) a[u] = fmaxf(a[u], __shfl_xor_sync(0xffffffffu, a[u], o));
  }
  // quotient d = lane mod 4U: group (u, half) = (d >> 2, (d >> 1) & 1), kind d & 1
  const int d = lane & (4 * U - 1);
  const int du = d >> 2, dh = (d >> 1) & 1;
  float ad = 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float t = __shfl_sync(0xffffffffu, a[u], 16 * dh);
    if (u == du) ad = t;
  }
  const bool kind = (d & 1) != 0;
  const float num = kind ? ad : 127.f, den = kind ? 127.f : ad;
  const float r = ad > 0.f ? __fdiv_rn(num, den) : 0.f;
  const int half = lane >> 4;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const size_t idx = base + static_cast<size_t>(u) * kCodecThreads;
    const int src = 4 * u + 2 * half;
    const float inv = __shfl_sync(0xffffffffu, r, src);
    const float sc = __shfl_sync(0xffffffffu, r, src + 1);
    uint32_t c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = code_byte(__fmul_rn(f[u][e], inv));
    if (idx < nvec) {
      uint2 o;
      o.x = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
      o.y = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
      q[idx] = o;
      if ((lane & (kVecPerGroup - 1)) == 0) scale[idx / kVecPerGroup] = sc;
    }
  }
}

template <int NP>
__global__ void __launch_bounds__(kCodecThreads)
codec_dequant_add_kernel(const uint4* __restrict__ own, const uint2* __restrict__ q,
                         const float* __restrict__ scale, size_t nvec, uint4* __restrict__ out) {
  pdl_wait_prior();
  const size_t base = static_cast<size_t>(blockIdx.x) * kCodecThreads * kDqUnroll + threadIdx.x;
  const size_t ngroups = nvec / kVecPerGroup;
  uint4 o[kDqUnroll];
  uint2 c[kDqUnroll][NP > 0 ? NP : 1];
  float s[kDqUnroll][NP > 0 ? NP : 1];
#pragma unroll
  for (int u = 0; u < kDqUnroll; ++u) {
    const size_t idx = base + static_cast<size_t>(u) * kCodecThreads;
    const bool ok = idx < nvec;
    o[u] = ok ? __ldcs(own + idx) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      c[u][p] = ok ? __ldcs(q + p * nvec + idx) : make_uint2(0, 0);
      s[u][p] = ok ? __ldg(scale + p * ngroups + idx / kVecPerGroup) : 0.f;
    }
  }
  pdl_launch_dependents();
#pragma unroll
  for (int u = 0; u < kDqUnroll; ++u) {
    const size_t idx = base + static_cast<size_t>(u) * kCodecThreads;
    float acc[8];
    bf16x8_to_f32(o[u], acc);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const uint32_t w[2] = {c[u][p].x, c[u][p].y};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int8_t v = static_cast<int8_t>((w[e >> 2] >> (8 * (e & 3))) & 0xFFu);
        acc[e] = __fadd_rn(acc[e], __fmul_rn(static_cast<float>(v), s[u][p]));
      }
    }
    if (idx < nvec) {
      uint4 r;
      r.x = pack_bf16x2(acc[0], acc[1]);
      r.y = pack_bf16x2(acc[2], acc[3]);
      r.z = pack_bf16x2(acc[4], acc[5]);
      r.w = pack_bf16x2(acc[6], acc[7]);
      out[idx] = r;
    }
  }
}

dim3 codec_grid(size_t nvec, int unroll) {
  const size_t per = static_cast<size_t>(kCodecThreads) * unroll;
  return dim3(static_cast<unsigned>((nvec + per - 1) / per));
}

template <int NP>
cudaError_t launch_dq(const uint16_t* own, const int8_t* q, const float* scale, size_t nvec,
                      uint16_t* out, cudaStream_t st) {
  return launch_pdl(codec_dequant_add_kernel<NP>, codec_grid(nvec, kDqUnroll), dim3(kCodecThreads), 0, st,
                    reinterpret_cast<const uint4*>(own), reinterpret_cast<const uint2*>(q), scale,
                    nvec, reinterpret_cast<uint4*>(out));
}

}  // namespace

cudaError_t launch_codec_quant(const uint16_t* x, int R, int H, int8_t* q, float* scale,
                               cudaStream_t st) {
  const size_t nvec = static_cast<size_t>(R) * H / 8;
  return launch_pdl(codec_quant_kernel<kQuantUnroll>, codec_grid(nvec, kQuantUnroll), dim3(kCodecThreads), 0, st,
                    reinterpret_cast<const uint4*>(x), nvec, reinterpret_cast<uint2*>(q), scale);
}

cudaError_t launch_codec_dequant_add(const uint16_t* own, const int8_t* q, const float* scale,
                                     int npeers, int R, int H, uint16_t* out, cudaStream_t st) {
  const size_t nvec = static_cast<size_t>(R) * H / 8;
  switch (npeers) {
    case 0: return launch_dq<0>(own, q, scale, nvec, out, st);
    case 1: return launch_dq<1>(own, q, scale, nvec, out, st);
    case 2: return launch_dq<2>(own, q, scale, nvec, out, st);
    case 3: return launch_dq<3>(own, q, scale, nvec, out, st);
    case 4: return launch_dq<4>(own, q, scale, nvec, out, st);
    case 5: return launch_dq<5>(own, q, scale, nvec, out, st);
    case 6: return launch_dq<6>(own, q, scale, nvec, out, st);
    case 7: return launch_dq<7>(own, q, scale, nvec, out, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tl
