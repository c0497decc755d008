// Helpers shared by the decode kernels (decode.cu, decode_fused_m.cu): the
// staged activations' dp4a order, the output store, the multi-token row
// layout and the distributed-shared-memory stores of the fused kernels.
#pragma once

#include "tl_internal.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace {

constexpr int kDecWarps = 8;

__device__ __forceinline__ void store_y(void* y, int y_dtype, size_t idx, float v) {
  if (y_dtype == TL_F32)
    static_cast<float*>(y)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// Permute 32 activation bytes (one chunk) into dp4a order; returns their sum.
__device__ __forceinline__ int permute_chunk(uint4 u0, uint4 u1, uint4& p0, uint4& p1) {
  p0.x = __byte_perm(u0.x, u0.z, 0x5140);
  p0.y = __byte_perm(u0.x, u0.z, 0x7362);
  p0.z = __byte_perm(u0.y, u0.w, 0x5140);
  p0.w = __byte_perm(u0.y, u0.w, 0x7362);
  p1.x = __byte_perm(u1.x, u1.z, 0x5140);
  p1.y = __byte_perm(u1.x, u1.z, 0x7362);
  p1.z = __byte_perm(u1.y, u1.w, 0x5140);
  p1.w = __byte_perm(u1.y, u1.w, 0x7362);
  int s = __dp4a(static_cast<int>(u0.x), 0x01010101, 0);
  s = __dp4a(static_cast<int>(u0.y), 0x01010101, s);
  s = __dp4a(static_cast<int>(u0.z), 0x01010101, s);
  s = __dp4a(static_cast<int>(u0.w), 0x01010101, s);
  s = __dp4a(static_cast<int>(u1.x), 0x01010101, s);
  s = __dp4a(static_cast<int>(u1.y), 0x01010101, s);
  s = __dp4a(static_cast<int>(u1.z), 0x01010101, s);
  s = __dp4a(static_cast<int>(u1.w), 0x01010101, s);
  return s;
}

// Row layout of the multi-token decode (2 <= MT <= 16, MT * K <= 72 K): RPW rows
// per warp, GR rows sharing each staged activation read, RC (row group, chunk)
// steps of weights in flight; SMEM bytes of staged activations.
template <int PL, int MT>
struct MTTraits {
  static constexpr int RPW = PL <= 8 ? 4 : 2;                    // rows per warp
  static constexpr int ROWS = kDecWarps * RPW;                   // rows per CTA
  // rows sharing one activation read: all 4 of a warp at MT = 4, 8 (M = 4: 15.0 -> 13.5 us,
  // M = 8: 20.8 -> 19.4 us at K = 5120; at MT = 2 the 4-row version measured 10.1 against 7.2 us)
  static constexpr int GR = MT >= 16 ? 1 : ((MT >= 4 && RPW == 4) ? 4 : 2);
  static constexpr int NG = RPW / GR;                            // row groups per warp
  // (group, chunk) steps in flight: 8 above K = 8192, as the M = 1 kernel there
  // (M = 4 at K = 17408: 19.2 -> 18.1 us), 3 below
  static constexpr int RC0 = PL > 8 ? 8 : 3;
  static constexpr int RC = PL * NG < RC0 ? PL * NG : RC0;
  static constexpr int QSTRIDE = ROWS + 4;
  static constexpr int LOG2MT = MT == 2 ? 1 : (MT == 4 ? 2 : (MT == 8 ? 3 : 4));
  static constexpr size_t SMEM = static_cast<size_t>(MT) * (PL * kBlock / 32) * 36;
};

// Distributed shared memory: the address of `p` in cluster CTA `rank`, and stores there.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer(uint32_t a, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t a, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

}  // namespace
}  // namespace tl
