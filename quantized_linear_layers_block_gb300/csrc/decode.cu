// K2: decode-time (M <= 32) ternary linear layer on the CUDA cores.
//
// Same integer accumulator and epilogue as the prefill GEMM of Qiita item
// ecc183fae033565af7cb §4 "効いた高速化"; the int8-activation GEMV with dp4a
// is the idea of §5 "効かなかったもの" (a dp4a decode GEMV), here computing
// exactly the quantised layer so that decode and prefill agree bit for bit.
//
// Kernels here: decode1_kernel (M = 1), decodem_kernel (2 <= M <= 16 while
// M * K <= 72 K), decode_kernel (the remaining M <= 32, K in shared-memory
// slabs) and decode1f_kernel (M = 1 with the rotation inside, in clusters);
// decode_fused_m.cu holds the fused multi-token kernel.
//
// Each CTA owns 32 consecutive output rows, 4 per warp (16 and 2 above
// K = 8192, where a row fills the register ring). Its first weight
// loads are issued at entry, before the kernel waits (programmatic dependent
// launch) for the activations of the preceding kernel, so the 2-bit weight
// stream of one layer overlaps the tail of the previous one. The packed
// weights, qT and sw are therefore read before that wait: they must be
// complete when the kernel is launched (tl_pack_weights at load time).
// The activations are staged in shared memory, permuted so that a 32-bit word
// of packed codes shifted by 2t and masked with 0x03030303 lines up byte for
// byte with activation word t:
//   e-bytes of (w >> 2t) & 0x03030303  ->  k = 2t, 2t+8, 2t+1, 2t+9
// dp4a(e, x) then gives sum (code + 1) x; the per-chunk activation sum is
// subtracted and the result multiplied by q[n, g] (integer, exact).
// Lane l of a warp owns the 32-code chunks l, l+32, ... of a row, so a
// warp-wide load of one row is fully coalesced 8-byte accesses.
#include "decode_common.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kRowsPerWarp = kRowsPerCta / kDecWarps;
constexpr int kQStride = kRowsPerCta + 4;   // padded: conflict-free q reads
constexpr size_t kSlabBudget = 96 * 1024;

__host__ __device__ constexpr int slab_k(int mt, int K) {
  // bytes per slab column: mt activations + mt/8 chunk sums (4 bytes per 32 codes)
  const size_t per_k = static_cast<size_t>(mt) * 9 / 8;
  size_t ks = kSlabBudget / per_k;
  ks = ks / kBlock * kBlock;
  if (ks < kBlock) ks = kBlock;
  return static_cast<int>(ks < static_cast<size_t>(K) ? ks : K);
}



// sum_k (code_k + 1) x_k over one 32-code chunk, starting from t.
__device__ __forceinline__ int dot_chunk(uint32_t wa, uint32_t wb, uint4 xa, uint4 xb, int t) {
  t = __dp4a(static_cast<int>(wa & 0x03030303u), static_cast<int>(xa.x), t);
  t = __dp4a(static_cast<int>((wa >> 2) & 0x03030303u), static_cast<int>(xa.y), t);
  t = __dp4a(static_cast<int>((wa >> 4) & 0x03030303u), static_cast<int>(xa.z), t);
  t = __dp4a(static_cast<int>((wa >> 6) & 0x03030303u), static_cast<int>(xa.w), t);
  t = __dp4a(static_cast<int>(wb & 0x03030303u), static_cast<int>(xb.x), t);
  t = __dp4a(static_cast<int>((wb >> 2) & 0x03030303u), static_cast<int>(xb.y), t);
  t = __dp4a(static_cast<int>((wb >> 4) & 0x03030303u), static_cast<int>(xb.z), t);
  t = __dp4a(static_cast<int>((wb >> 6) & 0x03030303u), static_cast<int>(xb.w), t);
  return t;
}

// The same sum with two masks per word: fields 0 and 2 (scale 1) and fields 1
// and 3 (scale 4, exact: P + Q/4 with Q a multiple of 4).
__device__ __forceinline__ int dot_chunk2(uint32_t wa, uint32_t wb, uint4 xa, uint4 xb, int t) {
  const uint32_t wa4 = wa >> 4, wb4 = wb >> 4;
  int p = t, q = 0;
  p = __dp4a(static_cast<int>(wa & 0x03030303u), static_cast<int>(xa.x), p);
  q = __dp4a(static_cast<int>(wa & 0x0C0C0C0Cu), static_cast<int>(xa.y), q);
  p = __dp4a(static_cast<int>(wa4 & 0x03030303u), static_cast<int>(xa.z), p);
  q = __dp4a(static_cast<int>(wa4 & 0x0C0C0C0Cu), static_cast<int>(xa.w), q);
  p = __dp4a(static_cast<int>(wb & 0x03030303u), static_cast<int>(xb.x), p);
  q = __dp4a(static_cast<int>(wb & 0x0C0C0C0Cu), static_cast<int>(xb.y), q);
  p = __dp4a(static_cast<int>(wb4 & 0x03030303u), static_cast<int>(xb.z), p);
  q = __dp4a(static_cast<int>(wb4 & 0x0C0C0C0Cu), static_cast<int>(xb.w), q);
  return p + (q >> 2);
}

// q of this CTA's rows for all groups (qT is group-major: 32 contiguous bytes per group).
__device__ __forceinline__ void stage_q(const int8_t* __restrict__ qT, int N, int G, int n0,
                                        int8_t* qs) {
  for (int i = threadIdx.x; i < G * (kRowsPerCta / 4); i += blockDim.x) {
    const int g = i / (kRowsPerCta / 4), r4 = i % (kRowsPerCta / 4);
    *reinterpret_cast<uint32_t*>(qs + g * kQStride + 4 * r4) =
        *reinterpret_cast<const uint32_t*>(qT + static_cast<size_t>(g) * N + n0 + 4 * r4);
  }
}

// ---------------------------------------------------------------- M = 1
// PL chunks of 32 codes per lane and row (K = 1024 PL). Fully unrolled over
// the warp's RPW rows and the PL chunks, so every ring slot is a register. The
// weight ring is chunk-major: RC chunk steps of all RPW rows in flight, so
// each staged activation chunk is read from shared memory once for all the
// warp's rows (reading it per row, 1 byte per code at 4 wavefronts per warp
// load, took as long as the arithmetic). The activations are staged once per
// CTA as two half-chunk arrays (conflict-free 16-byte reads) with their sums.
// Rows per warp: 4 while K <= 8192; 2 above, where one row fills the register
// ring and 4-row CTAs would leave too few warps per SM for short N (down_proj,
// K = 17408, N = 5120: 160 CTAs of 32 rows took 10.9 us, 320 of 16 take 8.2 us,
// 640 of 8 need 1.4 waves at 78 registers and took 10.0 us).
// While K <= 8192 the ring is one chunk step deep and the registers are capped
// for 5 CTAs per SM: a layer (544 CTAs at the gate+up shape) then leaves 216
// CTA slots free, so the next kernel's CTAs become resident and start their
// weight loads while this one computes (3 steps deep at 4 CTAs per SM, the
// rotate+GEMV pair took 7.7 us per layer; one step deep at 5 per SM, 7.0 us).
// CTAs per SM the M = 1 kernel's registers are capped for (0: no cap)
__host__ __device__ constexpr int m1_min_ctas(int pl) { return pl <= 8 ? 5 : 0; }

template <int PL>
struct M1Traits {
  static constexpr int RPW = PL <= 8 ? 4 : 2;                 // rows per warp
  static constexpr int ROWS = kDecWarps * RPW;                // rows per CTA
  static constexpr int RC = PL <= 8 ? 1 : 8;                  // chunk steps (of all RPW rows) in flight
  static constexpr int QSTRIDE = ROWS + 4;                    // padded q row: conflict-free reads
};

// The CTA's shared state of the M = 1 GEMV (as the fused kernel below holds
// it): the staged, permuted token and q.
template <int PL>
struct M1Smem {
  static constexpr int NC = PL * kBlock / 32;
  static constexpr int G = PL * kBlock / kGroup;
  uint4 xw0[NC];
  uint4 xw1[NC];
  int csum[NC];
  int8_t qs[G * M1Traits<PL>::QSTRIDE];
};

// Entry of an M = 1 CTA: the first RC chunk steps of the warp's rows into the
// register ring, then q of the CTA's rows (qT is group-major: ROWS contiguous
// bytes per group). Weights only, so it runs before the wait on the
// preceding kernel.
template <int PL>
__device__ __forceinline__ void m1_prologue(const uint32_t* __restrict__ packed,
                                            const int8_t* __restrict__ qT, int N, M1Smem<PL>& sm,
                                            uint2 (&ring)[M1Traits<PL>::RC][M1Traits<PL>::RPW]) {
  using T = M1Traits<PL>;
  constexpr int NC = M1Smem<PL>::NC, G = M1Smem<PL>::G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * T::ROWS;
  const uint2* pw = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * NC + lane;
  constexpr size_t kRowStep = static_cast<size_t>(kDecWarps) * NC;   // uint2 between a warp's rows
#pragma unroll
  for (int i = 0; i < T::RC; ++i) {
#pragma unroll
    for (int j = 0; j < T::RPW; ++j) ring[i][j] = __ldg(pw + j * kRowStep + i * 32);
  }
  pdl_launch_dependents();
  for (int i = tid; i < G * (T::ROWS / 4); i += blockDim.x) {
    const int g = i / (T::ROWS / 4), r4 = i % (T::ROWS / 4);
    *reinterpret_cast<uint32_t*>(sm.qs + g * T::QSTRIDE + 4 * r4) =
        *reinterpret_cast<const uint32_t*>(qT + static_cast<size_t>(g) * N + n0 + 4 * r4);
  }
}

// The GEMV of the CTA's rows from the staged token, and its epilogue.
template <int PL>
__device__ __forceinline__ void m1_gemv(const uint32_t* __restrict__ packed,
                                        const float* __restrict__ sw, float sx0, int N,
                                        const M1Smem<PL>& sm,
                                        uint2 (&ring)[M1Traits<PL>::RC][M1Traits<PL>::RPW],
                                        void* __restrict__ y, int y_dtype,
                                        int32_t* __restrict__ acc_dbg) {
  using T = M1Traits<PL>;
  constexpr int NC = M1Smem<PL>::NC;
  constexpr int RPW = T::RPW, RC = T::RC, QS = T::QSTRIDE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * T::ROWS;
  const uint2* pw = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * NC + lane;
  constexpr size_t kRowStep = static_cast<size_t>(kDecWarps) * NC;
  int acc[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) acc[k] = 0;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int c = i * 32 + lane;
    const uint4 xa = sm.xw0[c], xb = sm.xw1[c];      // read once for all the warp's rows
    const int cs = -sm.csum[c];
    const int8_t* qrow = sm.qs + (8 * i + (lane >> 2)) * QS + warp;
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const uint2 wv = ring[i % RC][k];
      if (i + RC < PL) ring[i % RC][k] = __ldg(pw + k * kRowStep + (i + RC) * 32);
      const int t = dot_chunk2(wv.x, wv.y, xa, xb, cs);
      acc[k] += static_cast<int>(qrow[kDecWarps * k]) * t;
    }
  }
  // the RPW sums together: exchange halves, then the remaining butterfly steps
  int tk = 0;
  constexpr int LOG2R = RPW == 1 ? 0 : (RPW == 2 ? 1 : 2);
#pragma unroll
  for (int st = 0; st < LOG2R; ++st) {
    const int half = RPW >> (st + 1);
    const int o = 16 >> st;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const int send = up ? acc[k] : acc[k + half];
      const int keep = up ? acc[k + half] : acc[k];
      acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) tk += half;
  }
#pragma unroll
  for (int o = 16 >> LOG2R; o > 0; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
  if ((lane & ((32 >> LOG2R) - 1)) == 0) {
    const int n = n0 + warp + kDecWarps * tk;
    if (acc_dbg != nullptr) acc_dbg[n] = acc[0];
    store_y(y, y_dtype, n, __fmul_rn(__fmul_rn(__int2float_rn(acc[0]), sw[n]), sx0));
  }
}

// decode1_kernel keeps its own copy of the prologue and the GEMV: built from
// the shared functions above it measured 4 % slower back to back (5.37 against
// 5.15 us at the gate+up shape), with the same results.
template <int PL>
__global__ void __launch_bounds__(kDecWarps * 32, m1_min_ctas(PL))
decode1_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
               const float* __restrict__ sw, const int8_t* __restrict__ xq,
               const float* __restrict__ sx, int N, void* __restrict__ y, int y_dtype,
               int32_t* __restrict__ acc_dbg) {
  constexpr int K = PL * kBlock;
  constexpr int G = K / kGroup;
  constexpr int NC = K / 32;                           // chunks per row
  constexpr int RPW = M1Traits<PL>::RPW;
  constexpr int ROWS = M1Traits<PL>::ROWS;
  constexpr int RC = M1Traits<PL>::RC;
  constexpr int QS = M1Traits<PL>::QSTRIDE;
  __shared__ __align__(16) uint4 xw0[NC];
  __shared__ __align__(16) uint4 xw1[NC];
  __shared__ int csum[NC];
  __shared__ __align__(16) int8_t qs[G * QS];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n0 = blockIdx.x * ROWS;
  const uint2* pw = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * NC + lane;
  constexpr size_t kRowStep = static_cast<size_t>(kDecWarps) * NC;   // uint2 between a warp's rows

  // chunk-major ring: RC chunk steps, each holding the chunk of all RPW rows
  uint2 ring[RC][RPW];
#pragma unroll
  for (int i = 0; i < RC; ++i) {
#pragma unroll
    for (int j = 0; j < RPW; ++j) ring[i][j] = __ldg(pw + j * kRowStep + i * 32);
  }
  pdl_launch_dependents();
  // q of this CTA's rows for all groups (qT is group-major: ROWS contiguous bytes per group)
  for (int i = tid; i < G * (ROWS / 4); i += blockDim.x) {
    const int g = i / (ROWS / 4), r4 = i % (ROWS / 4);
    *reinterpret_cast<uint32_t*>(qs + g * QS + 4 * r4) =
        *reinterpret_cast<const uint32_t*>(qT + static_cast<size_t>(g) * N + n0 + 4 * r4);
  }
  pdl_wait_prior();
  for (int c = tid; c < NC; c += blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(xq + 32 * c);
    uint4 p0, p1;
    csum[c] = permute_chunk(src[0], src[1], p0, p1);
    xw0[c] = p0;
    xw1[c] = p1;
  }
  __syncthreads();
  const float sx0 = sx[0];

  int acc[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) acc[k] = 0;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int c = i * 32 + lane;
    const uint4 xa = xw0[c], xb = xw1[c];            // read once for all the warp's rows
    const int cs = -csum[c];
    const int8_t* qrow = qs + (8 * i + (lane >> 2)) * QS + warp;
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const uint2 wv = ring[i % RC][k];
      if (i + RC < PL) ring[i % RC][k] = __ldg(pw + k * kRowStep + (i + RC) * 32);
      const int t = dot_chunk2(wv.x, wv.y, xa, xb, cs);
      acc[k] += static_cast<int>(qrow[kDecWarps * k]) * t;
    }
  }
  // the RPW sums together: exchange halves, then the remaining butterfly steps
  int tk = 0;
  constexpr int LOG2R = RPW == 1 ? 0 : (RPW == 2 ? 1 : 2);
#pragma unroll
  for (int st = 0; st < LOG2R; ++st) {
    const int half = RPW >> (st + 1);
    const int o = 16 >> st;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const int send = up ? acc[k] : acc[k + half];
      const int keep = up ? acc[k + half] : acc[k];
      acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) tk += half;
  }
#pragma unroll
  for (int o = 16 >> LOG2R; o > 0; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
  if ((lane & ((32 >> LOG2R) - 1)) == 0) {
    const int n = n0 + warp + kDecWarps * tk;
    if (acc_dbg != nullptr) acc_dbg[n] = acc[0];
    store_y(y, y_dtype, n, __fmul_rn(__fmul_rn(__int2float_rn(acc[0]), sw[n]), sx0));
  }
}

// ---------------------------------------------------------------- 2 <= M <= 16, small M * K
// The M = 1 kernel's layout for MT tokens (M rounded up to a power of two):
// the masked code words of a chunk are formed once per row and taken into dp4a
// with each token's staged activations (dynamic shared memory, MT * K * 9/8
// bytes, so MT * K is kept to 72 K); GR rows share each activation read (the
// reads cost MT bytes per code and bound the kernel when every row repeats them). A warp's MT row sums are reduced together: at
// each of log2(MT) exchange steps a lane keeps half of its tokens and adds the
// partner's half of the same tokens (MT - 1 shuffles), then the remaining
// 5 - log2(MT) butterfly steps finish the sum (instead of 5 MT shuffles).

template <int PL, int MT>
__global__ void __launch_bounds__(kDecWarps * 32)
decodem_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
               const float* __restrict__ sw, const int8_t* __restrict__ xq,
               const float* __restrict__ sx, int M, int N, void* __restrict__ y, int y_dtype,
               int32_t* __restrict__ acc_dbg) {
  using T = MTTraits<PL, MT>;
  constexpr int K = PL * kBlock;
  constexpr int G = K / kGroup;
  constexpr int NC = K / 32;
  constexpr int ROWS = T::ROWS, GR = T::GR, NG = T::NG, RC = T::RC, QS = T::QSTRIDE;
  extern __shared__ __align__(16) uint8_t dsm[];
  uint4* xw0 = reinterpret_cast<uint4*>(dsm);            // [MT][NC]
  uint4* xw1 = xw0 + MT * NC;                             // [MT][NC]
  int* csum = reinterpret_cast<int*>(xw1 + MT * NC);      // [MT][NC]
  __shared__ __align__(16) int8_t qs[G * QS];
  __shared__ float sxs[MT];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n0 = blockIdx.x * ROWS;
  const uint2* pw = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * NC + lane;
  constexpr size_t kRowStep = static_cast<size_t>(kDecWarps) * NC;

  // ring over the flattened (row group, chunk) steps t = g PL + i: GR rows' chunk i
  uint2 ring[RC][GR];
#pragma unroll
  for (int t = 0; t < RC; ++t) {
#pragma unroll
    for (int k = 0; k < GR; ++k)
      ring[t][k] = __ldg(pw + ((t / PL) * GR + k) * kRowStep + (t % PL) * 32);
  }
  pdl_launch_dependents();
  for (int i = tid; i < G * (ROWS / 4); i += blockDim.x) {
    const int g = i / (ROWS / 4), r4 = i % (ROWS / 4);
    *reinterpret_cast<uint32_t*>(qs + g * QS + 4 * r4) =
        *reinterpret_cast<const uint32_t*>(qT + static_cast<size_t>(g) * N + n0 + 4 * r4);
  }
  pdl_wait_prior();
  for (int i = tid; i < MT * NC; i += blockDim.x) {
    const int m = i / NC, c = i - m * NC;
    uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
    if (m < M) {
      const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<size_t>(m) * K + 32 * c);
      u0 = src[0];
      u1 = src[1];
    }
    uint4 p0, p1;
    csum[i] = permute_chunk(u0, u1, p0, p1);
    xw0[i] = p0;
    xw1[i] = p1;
  }
  if (tid < MT) sxs[tid] = tid < M ? sx[tid] : 0.f;
  __syncthreads();

#pragma unroll
  for (int g = 0; g < NG; ++g) {
    int acc[GR][MT];
#pragma unroll
    for (int k = 0; k < GR; ++k)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[k][m] = 0;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int t = g * PL + i;
      const int c = i * 32 + lane;
      uint32_t e[GR][8];
      int q[GR];
#pragma unroll
      for (int k = 0; k < GR; ++k) {
        const uint2 wv = ring[t % RC][k];
        if (t + RC < NG * PL)
          ring[t % RC][k] = __ldg(pw + (((t + RC) / PL) * GR + k) * kRowStep + ((t + RC) % PL) * 32);
        e[k][0] = wv.x & 0x03030303u;
        e[k][1] = (wv.x >> 2) & 0x03030303u;
        e[k][2] = (wv.x >> 4) & 0x03030303u;
        e[k][3] = (wv.x >> 6) & 0x03030303u;
        e[k][4] = wv.y & 0x03030303u;
        e[k][5] = (wv.y >> 2) & 0x03030303u;
        e[k][6] = (wv.y >> 4) & 0x03030303u;
        e[k][7] = (wv.y >> 6) & 0x03030303u;
        q[k] = qs[(8 * i + (lane >> 2)) * QS + warp + kDecWarps * (g * GR + k)];
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const uint4 xa = xw0[m * NC + c], xb = xw1[m * NC + c];   // one read for the GR rows
        const int cs = -csum[m * NC + c];
#pragma unroll
        for (int k = 0; k < GR; ++k) {
          int d = cs;
          d = __dp4a(static_cast<int>(e[k][0]), static_cast<int>(xa.x), d);
          d = __dp4a(static_cast<int>(e[k][1]), static_cast<int>(xa.y), d);
          d = __dp4a(static_cast<int>(e[k][2]), static_cast<int>(xa.z), d);
          d = __dp4a(static_cast<int>(e[k][3]), static_cast<int>(xa.w), d);
          d = __dp4a(static_cast<int>(e[k][4]), static_cast<int>(xb.x), d);
          d = __dp4a(static_cast<int>(e[k][5]), static_cast<int>(xb.y), d);
          d = __dp4a(static_cast<int>(e[k][6]), static_cast<int>(xb.z), d);
          d = __dp4a(static_cast<int>(e[k][7]), static_cast<int>(xb.w), d);
          acc[k][m] += q[k] * d;
        }
      }
    }
    // per row of the group: reduce-scatter over the tokens, then finish the lane's token
#pragma unroll
    for (int k = 0; k < GR; ++k) {
      int tm = 0;
#pragma unroll
      for (int st = 0; st < T::LOG2MT; ++st) {
        const int half = MT >> (st + 1);
        const int o = 16 >> st;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int h = 0; h < half; ++h) {
          const int send = up ? acc[k][h] : acc[k][h + half];
          const int keep = up ? acc[k][h + half] : acc[k][h];
          acc[k][h] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) tm += half;
      }
#pragma unroll
      for (int o = 16 >> T::LOG2MT; o > 0; o >>= 1) acc[k][0] += __shfl_xor_sync(0xffffffffu, acc[k][0], o);
      if ((lane & ((32 >> T::LOG2MT) - 1)) == 0 && tm < M) {
        const int n = n0 + warp + kDecWarps * (g * GR + k);
        const size_t idx = static_cast<size_t>(tm) * N + n;
        if (acc_dbg != nullptr) acc_dbg[idx] = acc[k][0];
        store_y(y, y_dtype, idx, __fmul_rn(__fmul_rn(__int2float_rn(acc[k][0]), sw[n]), sxs[tm]));
      }
    }
  }
}

// The four warps of rotating group g (named barrier 1 + g, 128 threads).
__device__ __forceinline__ void group_sync(int g) {
  if (g == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

// ---------------------------------------------------------------- M = 1, fused
// One launch for the whole layer at M = 1: the kernel takes the bf16 token and
// does the input-side rotation and the per-token quantisation itself (the
// arithmetic of tl_rotate_quant_act, so the result is the same bit for bit)
// before the M = 1 GEMV above (same rows per CTA). The grid runs in clusters
// of CS CTAs that share the token through distributed shared memory: in
// cluster rank r, group g of four warps rotates block b = g CS + r (each lane
// 8 elements: strides 1-4 in registers, 8-128 across lanes, 256 and 512
// between the group's warps through shared memory), pushes the block maximum
// to every CTA of the cluster, and after a cluster barrier quantises its
// block, permutes it into the dp4a order (one chunk per lane of the group's
// first warp) and pushes the chunks and their sums to every CTA of the
// cluster; a second barrier and the GEMV follow. So a token is rotated once
// per cluster, by CTAs that would otherwise wait, and no CTA reads a peer
// after the second barrier (each one's shared memory outlives every write
// into it). Registers are capped for 4 CTAs per SM, not 5: under the
// 48-register cap the rotation spills. Per-CTA timestamps inside a 64-layer
// graph put the pieces at: the wait on the preceding layer 0.5 us past its
// last CTA, the token's load and rotation up to the first cluster barrier
// 1.8 us, quantise + push up to the second 1.5 us, the GEMV 3-4 us; the
// two-launch pair (rotate + quantise, then decode1_kernel) spends the same
// ~3.6 us before its GEMV and stays slightly faster (7.2 against 8.2 us per
// layer). One warp per block (5 of a cluster's warps) measured 8.3 us; every
// CTA rotating the whole token itself (no cluster) 11.3 us, its 544 CTAs
// reading the same 10 KB of activations.


template <int PL, int CS>
__global__ void __launch_bounds__(kDecWarps * 32, 4)
decode1f_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
                const float* __restrict__ sw, const uint16_t* __restrict__ x,
                const int8_t* __restrict__ signs, int N, void* __restrict__ y, int y_dtype,
                int32_t* __restrict__ acc_dbg, int8_t* __restrict__ xq_out,
                float* __restrict__ sx_out) {
  static_assert(PL <= 2 * CS, "two rotating groups of four warps per CTA");
  __shared__ __align__(16) M1Smem<PL> sm;
  __shared__ __align__(16) float xs[2][2][4][256];   // [group][stride 256 / 512][warp][element]
  __shared__ __align__(16) int8_t xnat[2][kBlock];   // a group's quantised block, natural order
  __shared__ float gmax[2][4];
  __shared__ float bmax[PL];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint2 ring[M1Traits<PL>::RC][M1Traits<PL>::RPW];
  m1_prologue<PL>(packed, qT, N, sm, ring);
  pdl_wait_prior();

  // group g (warps 4 g .. 4 g + 3) of cluster rank r rotates block b = g CS + r;
  // warp w4 of the group holds the elements 256 w4 + 8 lane + e
  const uint32_t rank = cluster_ctarank();
  const int g = warp >> 2, w4 = warp & 3;
  const int b = g * CS + static_cast<int>(rank);
  const bool rot = b < PL;
  const int i0 = 256 * w4 + 8 * lane;
  float v[8];
  if (rot) {
    const uint4 raw = *reinterpret_cast<const uint4*>(x + b * kBlock + i0);
    const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
    if (signs != nullptr) {
      const uint2 sr = *reinterpret_cast<const uint2*>(signs + b * kBlock + i0);
      const uint32_t sg[2] = {sr.x, sr.y};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int8_t sgn = static_cast<int8_t>((sg[e >> 2] >> (8 * (e & 3))) & 0xFFu);
        if (sgn < 0) v[e] = -v[e];
      }
    }
    // strides 1, 2, 4 (registers), 8 .. 128 (lanes), 256, 512 (the group's
    // warps, through shared memory): the order and arithmetic of rotate_block_warp
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if ((e & h) == 0) fwht_bfly(v[e], v[e + h]);
      }
    }
#pragma unroll
    for (int t = 1; t < 32; t <<= 1) {
      const float sg = (lane & t) != 0 ? -1.f : 1.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = __fmaf_rn(v[e], sg, __shfl_xor_sync(0xffffffffu, v[e], t));
    }
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      float4* mine = reinterpret_cast<float4*>(&xs[g][st][w4][8 * lane]);
      mine[0] = make_float4(v[0], v[1], v[2], v[3]);
      mine[1] = make_float4(v[4], v[5], v[6], v[7]);
      group_sync(g);
      const float4* other = reinterpret_cast<const float4*>(&xs[g][st][w4 ^ (1 << st)][8 * lane]);
      const float4 o0 = other[0], o1 = other[1];
      const float o[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
      const bool upper = (w4 >> st) & 1;   // the upper warp of the pair keeps partner - own
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = upper ? __fsub_rn(o[e], v[e]) : __fadd_rn(v[e], o[e]);
    }
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = __fmul_rn(v[e], 0.03125f);
      am = fmaxf(am, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (lane == 0) gmax[g][w4] = am;
    group_sync(g);
    if (w4 == 0 && lane < CS) {
      const float bm = fmaxf(fmaxf(gmax[g][0], gmax[g][1]), fmaxf(gmax[g][2], gmax[g][3]));
      st_peer(peer_addr(&bmax[b], lane), bm);
    }
  }
  cluster_sync();
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) a = fmaxf(a, bmax[i]);
  const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
  const float sx0 = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
  if (rot) {
    int q8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) q8[e] = quant_i8(v[e], inv);
    uint2 o;
    o.x = (q8[0] & 0xFF) | ((q8[1] & 0xFF) << 8) | ((q8[2] & 0xFF) << 16) | ((q8[3] & 0xFF) << 24);
    o.y = (q8[4] & 0xFF) | ((q8[5] & 0xFF) << 8) | ((q8[6] & 0xFF) << 16) | ((q8[7] & 0xFF) << 24);
    *reinterpret_cast<uint2*>(&xnat[g][i0]) = o;
    if (xq_out != nullptr && blockIdx.x < CS)   // the first cluster writes xq_out
      *reinterpret_cast<uint2*>(xq_out + b * kBlock + i0) = o;
    group_sync(g);
    if (w4 == 0) {
      // lane c permutes chunk c of the block into the dp4a order and pushes it
      // with its sum to every CTA of the cluster
      const uint4* src = reinterpret_cast<const uint4*>(&xnat[g][32 * lane]);
      uint4 p0, p1;
      const int cs = permute_chunk(src[0], src[1], p0, p1);
      const int c = b * 32 + lane;
#pragma unroll
      for (int r = 0; r < CS; ++r) {
        st_peer(peer_addr(&sm.xw0[c], r), p0);
        st_peer(peer_addr(&sm.xw1[c], r), p1);
        st_peer(peer_addr(&sm.csum[c], r), cs);
      }
    }
  }
  if (sx_out != nullptr && blockIdx.x == 0 && tid == 0) sx_out[0] = sx0;
  cluster_sync();
  m1_gemv<PL>(packed, sw, sx0, N, sm, ring, y, y_dtype, acc_dbg);
}

// ---------------------------------------------------------------- 1 <= M <= 32
// MT tokens per pass (M rounded up to a power of two). A warp walks its
// (row, chunk) items in order and keeps PF weight loads in flight; the first
// PF are issued at entry. When MT * K does not fit in shared memory, K is
// processed in slabs and per-row partial sums are kept in shared memory.
template <int MT>
struct DecodeTraits {
  static constexpr int PF = MT <= 2 ? 16 : 8;
};

template <int MT>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
              const float* __restrict__ sw, const int8_t* __restrict__ xq,
              const float* __restrict__ sx, int M, int N, int K, int KS, void* __restrict__ y,
              int y_dtype, int32_t* __restrict__ acc_dbg) {
  constexpr int PF = DecodeTraits<MT>::PF;
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = K / kGroup;
  uint4* xw0 = reinterpret_cast<uint4*>(smem);                                    // [MT][KS/32]
  uint4* xw1 = reinterpret_cast<uint4*>(smem + static_cast<size_t>(MT) * KS / 2);  // [MT][KS/32]
  int32_t* csum = reinterpret_cast<int32_t*>(smem + static_cast<size_t>(MT) * KS);  // [MT][KS/32]
  int8_t* qs = reinterpret_cast<int8_t*>(smem + static_cast<size_t>(MT) * KS * 9 / 8);  // [G][kQStride]
  int32_t* part = reinterpret_cast<int32_t*>(
      smem + static_cast<size_t>(MT) * KS * 9 / 8 + ((static_cast<size_t>(G) * kQStride + 15) & ~size_t(15)));  // [32][MT]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n0 = blockIdx.x * kRowsPerCta;
  const int nslab = (K + KS - 1) / KS;
  const size_t row_step = static_cast<size_t>(kDecWarps) * (K / 32);   // uint2 between a warp's rows
  const uint2* prow0 = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * (K / 32) + lane;

  uint2 ring[PF];
  int per_lane = min(KS, K) / kBlock;
  int items = kRowsPerWarp * per_lane;
  // position of the next item to load (row slot, chunk)
  int prr = 0, pci = 0;
#pragma unroll
  for (int u = 0; u < PF; ++u) {
    if (u < items) {
      ring[u] = __ldg(prow0 + prr * row_step + pci * 32);
      if (++pci == per_lane) {
        pci = 0;
        ++prr;
      }
    }
  }
  pdl_launch_dependents();
  stage_q(qT, N, G, n0, qs);
  pdl_wait_prior();

  for (int sl = 0; sl < nslab; ++sl) {
    const int k0 = sl * KS;
    const int ks = min(KS, K - k0);
    const int nchunk = ks / 32;
    per_lane = nchunk / 32;  // ks is a multiple of 1024
    items = kRowsPerWarp * per_lane;
    const uint2* prow = prow0 + k0 / 32;
    if (sl > 0) {
      __syncthreads();  // previous slab fully consumed
      prr = 0;
      pci = 0;
#pragma unroll
      for (int u = 0; u < PF; ++u) {
        if (u < items) {
          ring[u] = __ldg(prow + prr * row_step + pci * 32);
          if (++pci == per_lane) {
            pci = 0;
            ++prr;
          }
        }
      }
    }
    for (int i = tid; i < MT * nchunk; i += blockDim.x) {
      const int m = i / nchunk, c = i % nchunk;
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (m < M) {
        const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<size_t>(m) * K + k0 + 32 * c);
        u0 = src[0];
        u1 = src[1];
      }
      uint4 p0, p1;
      csum[m * (KS / 32) + c] = permute_chunk(u0, u1, p0, p1);
      xw0[m * (KS / 32) + c] = p0;
      xw1[m * (KS / 32) + c] = p1;
    }
    __syncthreads();

    int acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0;
    int rr = 0, ci = 0;   // row slot and chunk of the item being consumed
    for (int jb = 0; jb < items; jb += PF) {
#pragma unroll
      for (int u = 0; u < PF; ++u) {
        if (jb + u < items) {
          const uint2 wv = ring[u];
          if (jb + u + PF < items) {
            ring[u] = __ldg(prow + prr * row_step + pci * 32);
            if (++pci == per_lane) {
              pci = 0;
              ++prr;
            }
          }
          const int r = warp + kDecWarps * rr;
          const int c = ci * 32 + lane;                  // chunk index within the slab
          const int q = qs[((k0 / kGroup) + (c >> 2)) * kQStride + r];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int t = dot_chunk(wv.x, wv.y, xw0[m * (KS / 32) + c], xw1[m * (KS / 32) + c],
                                    -csum[m * (KS / 32) + c]);
            acc[m] += q * t;
          }
          if (++ci == per_lane) {
            // row r of this slab is complete: reduce over the warp
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
            }
            int mine = 0;
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (lane == m) mine = acc[m];
            if (lane < MT) {
              if (sl > 0) mine += part[r * MT + lane];
              if (sl + 1 < nslab) {
                part[r * MT + lane] = mine;
              } else if (lane < M) {
                const int n = n0 + r;
                const size_t idx = static_cast<size_t>(lane) * N + n;
                if (acc_dbg != nullptr) acc_dbg[idx] = mine;
                store_y(y, y_dtype, idx, __fmul_rn(__fmul_rn(__int2float_rn(mine), sw[n]), sx[lane]));
              }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0;
            ci = 0;
            ++rr;
          }
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
  return launch_pdl(decode_kernel<MT>, dim3(N / kRowsPerCta), dim3(kDecWarps * 32), smem, st,
                    packed, qT, sw, xq, sx, M, N, K, KS, y, y_dtype, acc_dbg);
}

template <int PL>
cudaError_t launch_m1(const uint32_t* packed, const int8_t* qT, const float* sw, const int8_t* xq,
                      const float* sx, int N, void* y, int y_dtype, int32_t* acc_dbg,
                      cudaStream_t st) {
  return launch_pdl(decode1_kernel<PL>, dim3(N / M1Traits<PL>::ROWS), dim3(kDecWarps * 32), 0, st,
                    packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg);
}

template <int PL, int MT>
cudaError_t launch_mm(const uint32_t* packed, const int8_t* qT, const float* sw, const int8_t* xq,
                      const float* sx, int M, int N, void* y, int y_dtype, int32_t* acc_dbg,
                      cudaStream_t st) {
  using T = MTTraits<PL, MT>;
  if (T::SMEM > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(decodem_kernel<PL, MT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(T::SMEM));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(decodem_kernel<PL, MT>, dim3(N / T::ROWS), dim3(kDecWarps * 32), T::SMEM, st,
                    packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg);
}

// The multi-token kernel for MT * K <= 72 K and the instantiated K; else -1.
template <int MT>
int try_mm(const uint32_t* packed, const int8_t* qT, const float* sw, const int8_t* xq,
           const float* sx, int M, int N, int K, void* y, int y_dtype, int32_t* acc_dbg,
           cudaStream_t st, cudaError_t* err) {
  if (static_cast<long long>(MT) * K > 72 * 1024) return -1;
  switch (K / kBlock) {
    case 1: *err = launch_mm<1, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0;
    case 2: *err = launch_mm<2, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0;
    case 3: *err = launch_mm<3, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0;
    case 4: *err = launch_mm<4, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0;
    case 5:
      if constexpr (MT <= 8) { *err = launch_mm<5, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0; }
      return -1;
    case 8:
      if constexpr (MT <= 8) { *err = launch_mm<8, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0; }
      return -1;
    case 16:
      if constexpr (MT <= 4) { *err = launch_mm<16, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0; }
      return -1;
    case 17:
      if constexpr (MT <= 4) { *err = launch_mm<17, MT>(packed, qT, sw, xq, sx, M, N, y, y_dtype, acc_dbg, st); return 0; }
      return -1;
    default: return -1;
  }
}

template <int PL, int CS>
cudaError_t launch_m1f_cs(const uint32_t* packed, const int8_t* qT, const float* sw, const uint16_t* x,
                          const int8_t* signs, int N, void* y, int y_dtype, int32_t* acc_dbg,
                          int8_t* xq_out, float* sx_out, cudaStream_t st) {
  return launch_pdl_cluster(decode1f_kernel<PL, CS>, dim3(N / M1Traits<PL>::ROWS), dim3(kDecWarps * 32), 0,
                            st, CS, packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out);
}

// Clusters of 8 CTAs where the grid allows it, else 4 (N is a multiple of 128,
// so the grid N / 32 always is a multiple of 4).
template <int PL>
cudaError_t launch_m1f(const uint32_t* packed, const int8_t* qT, const float* sw, const uint16_t* x,
                       const int8_t* signs, int N, void* y, int y_dtype, int32_t* acc_dbg,
                       int8_t* xq_out, float* sx_out, cudaStream_t st) {
  const int grid = N / M1Traits<PL>::ROWS;
  if (grid % 8 == 0)
    return launch_m1f_cs<PL, 8>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
  if (grid % 4 == 0)
    return launch_m1f_cs<PL, 4>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const uint32_t* packed, const int8_t* qT, const float* sw,
                          const int8_t* xq, const float* sx, int M, int N, int K, void* y,
                          int y_dtype, int32_t* acc_dbg, cudaStream_t st) {
  if (M == 1) {
    switch (K / kBlock) {
      case 1: return launch_m1<1>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 2: return launch_m1<2>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 3: return launch_m1<3>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 4: return launch_m1<4>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 5: return launch_m1<5>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 8: return launch_m1<8>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 16: return launch_m1<16>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      case 17: return launch_m1<17>(packed, qT, sw, xq, sx, N, y, y_dtype, acc_dbg, st);
      default: break;
    }
  }
  cudaError_t err = cudaSuccess;
  if (M == 2 && try_mm<2>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st, &err) == 0) return err;
  if (M >= 3 && M <= 4 && try_mm<4>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st, &err) == 0) return err;
  if (M >= 5 && M <= 8 && try_mm<8>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st, &err) == 0) return err;
  if (M >= 9 && M <= 16 && try_mm<16>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st, &err) == 0) return err;
  if (M <= 1) return launch_mt<1>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 2) return launch_mt<2>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 4) return launch_mt<4>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 8) return launch_mt<8>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  if (M <= 16) return launch_mt<16>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
  return launch_mt<32>(packed, qT, sw, xq, sx, M, N, K, y, y_dtype, acc_dbg, st);
}

cudaError_t launch_decode_fused(const uint32_t* packed, const int8_t* qT, const float* sw,
                                const uint16_t* x, const int8_t* signs, int N, int K, void* y,
                                int y_dtype, int32_t* acc_dbg, int8_t* xq_out, float* sx_out,
                                cudaStream_t st) {
  switch (K / kBlock) {
    case 1: return launch_m1f<1>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 2: return launch_m1f<2>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 3: return launch_m1f<3>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 4: return launch_m1f<4>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 5: return launch_m1f<5>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 6: return launch_m1f<6>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 7: return launch_m1f<7>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    case 8: return launch_m1f<8>(packed, qT, sw, x, signs, N, y, y_dtype, acc_dbg, xq_out, sx_out, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tl
