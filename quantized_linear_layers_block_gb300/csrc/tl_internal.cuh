// Internal declarations shared by the library's translation units: launch
// functions of each kernel, the device status word, and thin inline-PTX
// wrappers for sm_103a (mbarrier, TMA, tcgen05). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/tl.h"

namespace tl {

// ----------------------------------------------------------------- limits
constexpr int kBlock = 1024;          // Hadamard block and integer-exact fp32 chunk
constexpr int kGroup = 128;           // columns per fp16 weight scale
constexpr int kMaxK = 32768;          // rotate_quant holds one warp per 1024-block
constexpr int kMaxDecodeM = 32;
constexpr size_t kNoAllocScratchBytes = TL_NOALLOC_SCRATCH_BYTES;

// Bounded device waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ----------------------------------------------------------------- status word
__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- launchers
struct PrefillArgs {
  const uint8_t* packed;
  const int8_t* qT;
  const float* sw;
  const uint16_t* xq;
  const float* sx;
  int M, N, K;
  void* y;
  int y_dtype;
  int32_t* acc_dbg;
  void* workspace;
  size_t ws_bytes;
  bool clear_workspace;   // zero the part of the workspace the call uses before the kernel
};

cudaError_t launch_pack(const int8_t* codes, const uint16_t* s, int N, int K, uint32_t* packed,
                        int8_t* qT, float* sw, int* status, cudaStream_t st);
cudaError_t launch_rotate_quant(const uint16_t* x, int M, int K, const int8_t* signs, void* xq,
                                int xq_dtype, float* sx, cudaStream_t st);
cudaError_t launch_decode(const uint32_t* packed, const int8_t* qT, const float* sw,
                          const int8_t* xq, const float* sx, int M, int N, int K, void* y,
                          int y_dtype, int32_t* acc_dbg, cudaStream_t st);
// Fused decode of 2 <= M <= 16 tokens (M rounded up to MT, MT * K <= 72 K, the
// multi-token kernel's K); *supported is false, and nothing is launched, otherwise.
cudaError_t launch_decode_fused_m(const uint32_t* packed, const int8_t* qT, const float* sw,
                                  const uint16_t* x, const int8_t* signs, int M, int N, int K,
                                  void* y, int y_dtype, int32_t* acc_dbg, int8_t* xq_out,
                                  float* sx_out, cudaStream_t st, bool* supported);
// M = 1 decode with the rotation and quantisation of x done in each CTA (K <= 8192).
cudaError_t launch_decode_fused(const uint32_t* packed, const int8_t* qT, const float* sw,
                                const uint16_t* x, const int8_t* signs, int N, int K, void* y,
                                int y_dtype, int32_t* acc_dbg, int8_t* xq_out, float* sx_out,
                                cudaStream_t st);
constexpr int kMaxFusedDecodeK = 8192;
constexpr long long kMaxFusedMK = 72 * 1024;   // fused decode of M >= 2 tokens: MT * K staged
constexpr int kMaxCodecPeers = 7;
constexpr int kMaxF32ActM = 4;            // tokens of the float-activation decode
constexpr int kMaxF32ActMK = 36864;       // M * K bound: the staged fp32 activations fit shared memory
cudaError_t launch_rotate(const uint16_t* x, int M, int K, const int8_t* signs, float* xr,
                          cudaStream_t st);
cudaError_t launch_decode_f32act(const uint8_t* packed, const uint16_t* s, const float* xr, int M,
                                 int N, int K, void* y, int y_dtype, cudaStream_t st);
cudaError_t launch_codec_quant(const uint16_t* x, int R, int H, int8_t* q, float* scale,
                               cudaStream_t st);
cudaError_t launch_codec_dequant_add(const uint16_t* own, const int8_t* q, const float* scale,
                                     int npeers, int R, int H, uint16_t* out, cudaStream_t st);
size_t prefill_workspace_bytes(int M, int N, int K, int num_sms);
// True when the problem has fewer output tiles than SMs, so that splitting K
// is what keeps the GPU busy (not only the last, partial round).
bool prefill_split_required(int M, int N, int num_sms);
// Returns TL_OK or a tl_status; *cerr receives the CUDA error when TL_ECUDA.
int launch_prefill(const PrefillArgs& a, int* status, cudaStream_t st, cudaError_t* cerr);
// Device address (this device) of the library-owned split-K scratch array of
// kNoAllocScratchBytes; the first call on a device looks it up.
int prefill_noalloc_scratch(void** ptr);

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable), and a 2-D
// tiled tensor map over a row-major array of `outer` rows of `row_bytes`.
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn();
bool make_map_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, CUtensorMapDataType dt,
                 const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

// Tensor-core decode (1 <= M <= 32; xq the fp16 image of the int8 codes, [M, K]).
cudaError_t launch_decode_tc(const uint8_t* packed, const int8_t* qT, const float* sw,
                             const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                             int y_dtype, int32_t* acc_dbg, int* status, cudaStream_t st);

// Launch with programmatic stream serialization (PDL) enabled and, when
// cluster > 1, thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t st, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, st, 1, args...);
}

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy accesses (a TMA copy) that another thread issues after
// synchronising with it: required before releasing a shared-memory buffer
// that was read with ordinary loads to a producer that refills it by TMA.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up (returns
// false) when *abort becomes non-zero or after limit_ns (kWaitLimitNs).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// independent prologue now / wait until the previous kernel has completed.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---- tcgen05 (5th-generation tensor core, tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, repeated 32 times along the columns: each thread of the
// warp writes 32 consecutive columns of its own lane.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor (sm_100 family): K-major operand stored by a
// TMA SWIZZLE_128B load, i.e. rows of 128 bytes, 8-row (1024-byte) atoms.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);       // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1u) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7) | (0u << 10)                    // A, B format: f16
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// ---- input-side rotation of one 1024-column block by one warp
// Lane l holds the 32 elements i = 256 j + 8 l + e (j = 0..3, e = 0..7),
// loaded as four coalesced 16-byte vectors. Butterfly strides 1, 2, 4 act on e
// (registers), 8..128 on the lane index (warp shuffles), 256 and 512 on j
// (registers): the stages run in the order 1, 2, 4, ..., 512, each butterfly
// one fp32 add and one subtract, then the exact 1/32 scale. Returns the lane's
// largest |value|.
__device__ __forceinline__ void fwht_bfly(float& a, float& b) {
  const float s = __fadd_rn(a, b);
  const float d = __fsub_rn(a, b);
  a = s;
  b = d;
}

__device__ __forceinline__ float rotate_block_warp(const uint16_t* __restrict__ xb,
                                                   const int8_t* __restrict__ sb, int lane,
                                                   float (&v)[4][8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i0 = 256 * j + 8 * lane;
    const uint4 raw = *reinterpret_cast<const uint4*>(xb + i0);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
      v[j][e] = __uint_as_float(bits << 16);
    }
    if (sb != nullptr) {
      const uint2 sraw = *reinterpret_cast<const uint2*>(sb + i0);
      const uint32_t sg[2] = {sraw.x, sraw.y};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int8_t sgn = static_cast<int8_t>((sg[e >> 2] >> (8 * (e & 3))) & 0xFFu);
        if (sgn < 0) v[j][e] = -v[j][e];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if ((e & h) == 0) fwht_bfly(v[j][e], v[j][e + h]);
      }
    }
  }
#pragma unroll
  for (int t = 1; t < 32; t <<= 1) {
    // o - v on the upper lane of the pair, v + o on the lower: v * (+-1) + o,
    // exact before its one rounding, so bit for bit the subtract or the add
    const float sg = (lane & t) != 0 ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[j][e], t);
        v[j][e] = __fmaf_rn(v[j][e], sg, o);
      }
    }
  }
#pragma unroll
  for (int h = 1; h < 4; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((j & h) == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) fwht_bfly(v[j][e], v[j + h][e]);
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[j][e] = __fmul_rn(v[j][e], 0.03125f);
      amax = fmaxf(amax, fabsf(v[j][e]));
    }
  }
  return amax;
}

// Expansion of packed codes into the fp16 pairs code * q (expand_word below).
// The five (magic | magic << 16) words it ors into the fields are made once
// into registers: a LOP3 takes one immediate, and with both its mask and its
// magic as constants the compiler spent an extra instruction per pair on the
// second (the prefill kernel: 11 M fewer instructions per launch, 122.9 ->
// 120.0 us at the gate+up shape with 512 tokens).
struct ExpandMagic {
  uint32_t m[5];
};
__device__ __forceinline__ ExpandMagic expand_magic() {
  // the fp16 exponent fields (25 - 2 jj) << 10 in both halves
  ExpandMagic e;
  asm volatile("mov.b32 %0, 0x64006400;" : "=r"(e.m[0]));
  asm volatile("mov.b32 %0, 0x5C005C00;" : "=r"(e.m[1]));
  asm volatile("mov.b32 %0, 0x54005400;" : "=r"(e.m[2]));
  asm volatile("mov.b32 %0, 0x4C004C00;" : "=r"(e.m[3]));
  asm volatile("mov.b32 %0, 0x44004400;" : "=r"(e.m[4]));
  return e;
}
template <int JJ>
__device__ __forceinline__ uint32_t field_pair(uint32_t src, uint32_t magic2) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(src), "n"(0x00030003u << (2 * JJ)), "r"(magic2));
  return d;
}
// Expand one packed word (16 codes, layout of tl.h) into 8 fp16 pairs code*q.
// The 2-bit field e (= code + 1) is dropped into the mantissa of an fp16 whose
// exponent makes the value 2^E + e exactly; subtracting 2^E + 1 leaves the code
// in {-1, 0, +1} and one multiply by q gives code * q, all exact.
__device__ __forceinline__ void expand_word(uint32_t w, __half2 q2, uint32_t* out, const ExpandMagic& em) {
  const __half2 c0 = __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401));  // 1025
  const __half2 c1 = __halves2half2(__ushort_as_half(0x5C04), __ushort_as_half(0x5C04));  // 257
  const __half2 c2 = __halves2half2(__ushort_as_half(0x5410), __ushort_as_half(0x5410));  // 65
  const __half2 c3 = __halves2half2(__ushort_as_half(0x4C40), __ushort_as_half(0x4C40));  // 17
  const __half2 c4 = __halves2half2(__ushort_as_half(0x4500), __ushort_as_half(0x4500));  // 5
  const __half2 cs[5] = {c0, c1, c2, c3, c4};
  const uint32_t w10 = w >> 10;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int jj = j < 5 ? j : j - 5;
    const uint32_t src = j < 5 ? w : w10;
    uint32_t bits;
    switch (jj) {
      case 0: bits = field_pair<0>(src, em.m[0]); break;
      case 1: bits = field_pair<1>(src, em.m[1]); break;
      case 2: bits = field_pair<2>(src, em.m[2]); break;
      case 3: bits = field_pair<3>(src, em.m[3]); break;
      default: bits = field_pair<4>(src, em.m[4]); break;
    }
    __half2 h = *reinterpret_cast<const __half2*>(&bits);
    h = __hmul2(__hsub2(h, cs[jj]), q2);
    out[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Symmetric int8 code of one rotated value: clamp(rne(fl32(v inv)), -127, 127).
__device__ __forceinline__ int quant_i8(float v, float inv) {
  const int t = __float2int_rn(__fmul_rn(v, inv));
  return max(-127, min(127, t));
}

}  // namespace tl
