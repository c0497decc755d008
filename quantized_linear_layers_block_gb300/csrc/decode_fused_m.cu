// Fused decode for 2 <= M <= 16 tokens (M rounded up to MT, MT * K <= 72 K):
// the input-side rotation and per-token quantisation of tl_rotate_quant_act
// (Qiita item ecc183fae033565af7cb: 前提 for the block Hadamard rotation, §4
// for the per-token int8) done inside the multi-token dp4a GEMV (§5), bit for
// bit the result of the two launches.
//
// The grid runs in clusters of 4 CTAs with the multi-token GEMV's rows. The
// cluster shares the tokens through distributed shared memory:
//   1. The M x K/1024 (token, block) rotations are dealt over the cluster's
//      warps. A warp rotates its block in registers (the arithmetic of the
//      rotation kernel), keeps the fp32 result in its CTA's shared memory and
//      pushes the block's maximum |value| to every CTA of the cluster.
//   2. After a cluster barrier every CTA has every token's maximum, so the
//      warp quantises its block with the token's scale, permutes each 32-code
//      chunk into the dp4a order and pushes the chunks and their sums into the
//      staged activations of every CTA of the cluster.
//   3. After a second barrier the GEMV of the multi-token decode kernel runs
//      on the staged activations.
// No CTA reads a peer after the second barrier, so every write into a CTA's
// shared memory lands before that CTA can exit.
#include "decode_common.cuh"

namespace tl {
namespace {

constexpr int kFusedCluster = 4;

template <int PL, int MT>
struct FusedMTraits {
  static constexpr int TASKS = MT * PL;                                    // (token, block) pairs
  static constexpr int TPC = (TASKS + kFusedCluster - 1) / kFusedCluster;  // per CTA, at most
  // staged activations, then the CTA's rotated fp32 blocks
  static constexpr size_t XF_OFF = MTTraits<PL, MT>::SMEM;
  static constexpr size_t SMEM = XF_OFF + static_cast<size_t>(TPC) * kBlock * sizeof(float);
};

template <int PL, int MT>
__global__ void __launch_bounds__(kDecWarps * 32)
decodemf_kernel(const uint32_t* __restrict__ packed, const int8_t* __restrict__ qT,
                const float* __restrict__ sw, const uint16_t* __restrict__ x,
                const int8_t* __restrict__ signs, int M, int N, void* __restrict__ y, int y_dtype,
                int32_t* __restrict__ acc_dbg, int8_t* __restrict__ xq_out,
                float* __restrict__ sx_out) {
  using T = MTTraits<PL, MT>;
  using F = FusedMTraits<PL, MT>;
  constexpr int K = PL * kBlock;
  constexpr int G = K / kGroup;
  constexpr int NC = K / 32;
  constexpr int CS = kFusedCluster;
  constexpr int ROWS = T::ROWS, GR = T::GR, NG = T::NG, RC = T::RC, QS = T::QSTRIDE;
  extern __shared__ __align__(16) uint8_t dsm[];
  uint4* xw0 = reinterpret_cast<uint4*>(dsm);            // [MT][NC]
  uint4* xw1 = xw0 + MT * NC;                             // [MT][NC]
  int* csum = reinterpret_cast<int*>(xw1 + MT * NC);      // [MT][NC]
  float* xf = reinterpret_cast<float*>(dsm + F::XF_OFF);  // [TPC][1024]
  __shared__ __align__(16) int8_t qs[G * QS];
  __shared__ __align__(16) int8_t xnat[kDecWarps][kBlock];   // a warp's quantised block
  __shared__ float bmax[MT][PL];
  __shared__ float sxs[MT];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n0 = blockIdx.x * ROWS;
  const uint2* pw = reinterpret_cast<const uint2*>(packed) + static_cast<size_t>(n0 + warp) * NC + lane;
  constexpr size_t kRowStep = static_cast<size_t>(kDecWarps) * NC;

  // weights first (they do not depend on the preceding kernel), as the GEMV kernel does
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
  // padding tokens (m >= M) stage zeros and scale 0, locally
  for (int i = tid; i < (MT - M) * NC; i += blockDim.x) {
    const int j = M * NC + i;
    xw0[j] = make_uint4(0, 0, 0, 0);
    xw1[j] = make_uint4(0, 0, 0, 0);
    csum[j] = 0;
  }
  pdl_wait_prior();

  // 1. rotations: local task j of cluster rank r is task t = r + CS j, token t / PL, block t % PL
  const int rank = static_cast<int>(cluster_ctarank());
  for (int j = warp; j < F::TPC; j += kDecWarps) {
    const int t = rank + CS * j;
    const int m = t / PL, b = t - m * PL;
    if (t >= F::TASKS || m >= M) continue;
    float v[4][8];
    float am = rotate_block_warp(x + static_cast<size_t>(m) * K + b * kBlock,
                                 signs == nullptr ? nullptr : signs + b * kBlock, lane, v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    float* blk = xf + static_cast<size_t>(j) * kBlock;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float4* d = reinterpret_cast<float4*>(blk + 256 * jj + 8 * lane);
      d[0] = make_float4(v[jj][0], v[jj][1], v[jj][2], v[jj][3]);
      d[1] = make_float4(v[jj][4], v[jj][5], v[jj][6], v[jj][7]);
    }
    if (lane < CS) st_peer(peer_addr(&bmax[m][b], lane), am);
  }
  cluster_sync();

  // every token's scale from its block maxima
  if (tid < MT) {
    float a = 0.f;
    if (tid < M) {
#pragma unroll
      for (int b = 0; b < PL; ++b) a = fmaxf(a, bmax[tid][b]);
    }
    const float s = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
    sxs[tid] = s;
    if (sx_out != nullptr && blockIdx.x == 0 && tid < M) sx_out[tid] = s;
  }

  // 2. quantise the warp's blocks and push the permuted chunks to every CTA of the cluster
  for (int j = warp; j < F::TPC; j += kDecWarps) {
    const int t = rank + CS * j;
    const int m = t / PL, b = t - m * PL;
    if (t >= F::TASKS || m >= M) continue;
    float a = 0.f;
#pragma unroll
    for (int bb = 0; bb < PL; ++bb) a = fmaxf(a, bmax[m][bb]);
    const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
    const float* blk = xf + static_cast<size_t>(j) * kBlock;
    const bool out = xq_out != nullptr && blockIdx.x < CS;   // the first cluster writes xq_out
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const float4* s4 = reinterpret_cast<const float4*>(blk + 256 * jj + 8 * lane);
      const float4 f0 = s4[0], f1 = s4[1];
      const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      int q8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) q8[e] = quant_i8(f[e], inv);
      uint2 o;
      o.x = (q8[0] & 0xFF) | ((q8[1] & 0xFF) << 8) | ((q8[2] & 0xFF) << 16) | ((q8[3] & 0xFF) << 24);
      o.y = (q8[4] & 0xFF) | ((q8[5] & 0xFF) << 8) | ((q8[6] & 0xFF) << 16) | ((q8[7] & 0xFF) << 24);
      *reinterpret_cast<uint2*>(&xnat[warp][256 * jj + 8 * lane]) = o;
      if (out)
        *reinterpret_cast<uint2*>(xq_out + static_cast<size_t>(m) * K + b * kBlock + 256 * jj + 8 * lane) = o;
    }
    __syncwarp();
    const uint4* src = reinterpret_cast<const uint4*>(&xnat[warp][32 * lane]);
    uint4 p0, p1;
    const int cs = permute_chunk(src[0], src[1], p0, p1);
    __syncwarp();                                          // xnat is reused by the warp's next block
    const int c = m * NC + b * 32 + lane;
#pragma unroll
    for (int r = 0; r < CS; ++r) {
      st_peer(peer_addr(&xw0[c], r), p0);
      st_peer(peer_addr(&xw1[c], r), p1);
      st_peer(peer_addr(&csum[c], r), cs);
    }
  }
  cluster_sync();

  // 3. the multi-token GEMV on the staged tokens
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
        const uint4 xa = xw0[m * NC + c], xb = xw1[m * NC + c];
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

template <int PL, int MT>
cudaError_t launch_mf(const uint32_t* packed, const int8_t* qT, const float* sw, const uint16_t* x,
                      const int8_t* signs, int M, int N, void* y, int y_dtype, int32_t* acc_dbg,
                      int8_t* xq_out, float* sx_out, cudaStream_t st) {
  constexpr size_t smem = FusedMTraits<PL, MT>::SMEM;
  const cudaError_t e = cudaFuncSetAttribute(decodemf_kernel<PL, MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // N is a multiple of 128, so the grid (N / 32 or N / 16 CTAs) is a multiple of the cluster
  return launch_pdl_cluster(decodemf_kernel<PL, MT>, dim3(N / MTTraits<PL, MT>::ROWS),
                            dim3(kDecWarps * 32), smem, st, kFusedCluster, packed, qT, sw, x, signs,
                            M, N, y, y_dtype, acc_dbg, xq_out, sx_out);
}

template <int MT>
int try_mf(const uint32_t* packed, const int8_t* qT, const float* sw, const uint16_t* x,
           const int8_t* signs, int M, int N, int K, void* y, int y_dtype, int32_t* acc_dbg,
           int8_t* xq_out, float* sx_out, cudaStream_t st, cudaError_t* err) {
  if (static_cast<long long>(MT) * K > kMaxFusedMK) return -1;
#define TL_MF(PLV)                                                                                 \
  *err = launch_mf<PLV, MT>(packed, qT, sw, x, signs, M, N, y, y_dtype, acc_dbg, xq_out, sx_out, st); \
  return 0
  switch (K / kBlock) {
    case 1: TL_MF(1);
    case 2: TL_MF(2);
    case 3: TL_MF(3);
    case 4: TL_MF(4);
    case 5: if constexpr (MT <= 8) { TL_MF(5); } return -1;
    case 8: if constexpr (MT <= 8) { TL_MF(8); } return -1;
    case 16: if constexpr (MT <= 4) { TL_MF(16); } return -1;
    case 17: if constexpr (MT <= 4) { TL_MF(17); } return -1;
    default: return -1;
  }
#undef TL_MF
}

}  // namespace

cudaError_t launch_decode_fused_m(const uint32_t* packed, const int8_t* qT, const float* sw,
                                  const uint16_t* x, const int8_t* signs, int M, int N, int K,
                                  void* y, int y_dtype, int32_t* acc_dbg, int8_t* xq_out,
                                  float* sx_out, cudaStream_t st, bool* supported) {
  cudaError_t err = cudaSuccess;
  int r = -1;
  if (M == 2) r = try_mf<2>(packed, qT, sw, x, signs, M, N, K, y, y_dtype, acc_dbg, xq_out, sx_out, st, &err);
  else if (M <= 4) r = try_mf<4>(packed, qT, sw, x, signs, M, N, K, y, y_dtype, acc_dbg, xq_out, sx_out, st, &err);
  else if (M <= 8) r = try_mf<8>(packed, qT, sw, x, signs, M, N, K, y, y_dtype, acc_dbg, xq_out, sx_out, st, &err);
  else if (M <= 16) r = try_mf<16>(packed, qT, sw, x, signs, M, N, K, y, y_dtype, acc_dbg, xq_out, sx_out, st, &err);
  *supported = r == 0;
  return err;
}

}  // namespace tl
