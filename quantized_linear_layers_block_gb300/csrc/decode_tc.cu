// K2 on the tensor cores: the decode-time (1 <= M <= 32 tokens) ternary linear
// layer as an exact integer GEMM on mma.sync with fp16 operands.
//
// Qiita item ecc183fae033565af7cb §4 "効いた高速化" defines the quantised layer
// (acc[m,n] = sum_k xq[m,k] code[n,k] q[n,k/128], then the row and token
// rescale); §5 "効かなかったもの" is the decode GEMV it serves. The result is
// the same int32 accumulator, bit for bit, as the dp4a decode and the prefill.
//
// mma.sync.m16n8k16 (fp16 x fp16 -> fp32), 16 weight rows x 8 tokens per MMA:
//   A: the packed 2-bit codes of the rows, turned in registers into the fp16
//      pairs code q (the prefill's magic-number expansion: exact), so q rides
//      in the operand and no correction follows the MMA;
//   B: the fp16 image of the int8 codes (tl_rotate_quant_act, TL_F16), read as
//      it lies in memory: thread t of a fragment takes the columns
//      16 t + 64 h + 4 i + (0..3) of a 128-column group (h = 0, 1; i = 0..3),
//      and A's pairs are taken from packed words t and t + 4 of the group in
//      the same order.
// Every product |x w| <= 127 * 127 is exact in fp32 and every partial sum of at
// most 1024 columns is an integer below 2^24, so each warp sums eight groups
// in fp32 and then adds them, converted, to int32 totals: exact.
//
// Work: a CTA owns 16 * rbc weight rows and a range of the 128-column groups
// (a cluster of cs CTAs splits K; their partial sums meet in the first CTA's
// shared memory through distributed shared memory). One producer warp moves
// slabs of gs groups into a ring of shared-memory buffers: the weights and q
// by TMA tensor copies issued before the kernel waits for the preceding one
// (programmatic dependent launch), each token's activations by a bulk copy
// after (lane m of the producer warp issues token m's). Eight consumer warps
// each own one row block and one part of every slab's groups (kp = 8 / rbc
// parts).
#include "decode_common.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace {

constexpr int kTcConsumers = 8;
constexpr int kTcThreads = (kTcConsumers + 1) * 32;
constexpr int kTcMaxBuffers = 6;

struct TcPlan {
  int rbc;              // 16-row blocks per CTA
  int kp;               // consumer warps per row block (K parts of a slab)
  int cs;               // CTAs per cluster, splitting the groups
  int gs;               // groups per slab (odd: conflict-free weight reads)
  int sb;               // slab buffers
  uint32_t buf_bytes;   // bytes per slab buffer
  uint32_t off_q, off_b;   // offsets inside a buffer (weights at 0)
  uint32_t b_pitch;     // bytes between two tokens' activations in a buffer (16 mod 128)
  uint32_t red_off;     // int32 partial sums [rows][MP4]
  uint32_t bar_off;     // mbarriers full[sb], empty[sb], then the abort flag
  uint32_t smem;        // dynamic shared memory (before 1024-byte alignment)
};

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void red_add_peer(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 2)
decode_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_q,
                 const uint16_t* __restrict__ xq, const float* __restrict__ sw,
                 const float* __restrict__ sx, int M, int N, int K, TcPlan p, void* __restrict__ y,
                 int y_dtype, int32_t* __restrict__ acc_dbg, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned, as an offset into the shared array (shared loads)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int G = K / kGroup;
  const int MP4 = (M + 3) & ~3;
  const int rows = 16 * p.rbc;
  int32_t* red = reinterpret_cast<int32_t*>(smem + p.red_off);
  const uint32_t bar0 = sbase + p.bar_off;
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (p.sb + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.bar_off + 16 * p.sb);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = p.cs > 1 ? cluster_ctarank() : 0u;
  const int row0 = static_cast<int>(blockIdx.x / p.cs) * rows;
  const int gb = static_cast<int>((static_cast<long long>(crank) * G) / p.cs);
  const int ge = static_cast<int>((static_cast<long long>(crank + 1) * G) / p.cs);
  const int nslab = (ge - gb + p.gs - 1) / p.gs;
  const uint32_t wbytes = static_cast<uint32_t>(rows) * p.gs * 32;
  const uint32_t qbytes = static_cast<uint32_t>(rows) * p.gs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.sb; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), kTcConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < rows * MP4; i += blockDim.x) red[i] = 0;
  __syncthreads();
  // every CTA of the cluster has started and cleared its sums before any adds into a peer
  if (p.cs > 1) cluster_sync();

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(status, TL_ETIMEOUT);
  };
  // groups [g0, g0 + n) of slab s
  auto slab_groups = [&](int s, int* g0) {
    *g0 = gb + s * p.gs;
    const int left = ge - *g0;
    return left < p.gs ? left : p.gs;
  };

  if (warp == kTcConsumers) {
    // ------------------------------------------------------------- producer
    // the whole warp runs the loop; one elected lane issues the weight copies
    // and lane m issues token m's activation copy
    uint32_t elected;
    asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(elected));
    {
      if (elected) {
        tma_prefetch_desc(&map_w);
        tma_prefetch_desc(&map_q);
      }
      auto issue_w = [&](int s) {
        int g0;
        const int n = slab_groups(s, &g0);
        const int b = s % p.sb;
        const uint32_t buf = sbase + b * p.buf_bytes;
        if (elected) {
          mbar_arrive_expect_tx(full(b), wbytes + qbytes + static_cast<uint32_t>(M) * n * 256);
          tma_load_2d(buf, &map_w, g0 * 32, row0, full(b));
          tma_load_2d(buf + p.off_q, &map_q, row0, g0, full(b));
        }
        __syncwarp();
      };
      auto issue_x = [&](int s) {
        int g0;
        const int n = slab_groups(s, &g0);
        const int b = s % p.sb;
        const uint32_t dst = sbase + b * p.buf_bytes + p.off_b;
        for (int m = lane; m < M; m += 32)
          bulk_g2s(dst + m * p.b_pitch, xq + static_cast<size_t>(m) * K + g0 * kGroup, n * 256,
                   full(b));
        __syncwarp();
      };
      const int pre = nslab < p.sb ? nslab : p.sb;
      // weights and q only: they do not come from the preceding kernel
      for (int s = 0; s < pre; ++s) issue_w(s);
      if (elected) pdl_launch_dependents();
      pdl_wait_prior();
      for (int s = 0; s < pre; ++s) issue_x(s);
      int issued = pre;
      for (int s = pre; s < nslab; ++s) {
        const int b = s % p.sb;
        if (!__all_sync(0xffffffffu, mbar_wait(empty(b), static_cast<uint32_t>((s / p.sb) - 1) & 1u, abort_flag))) {
          fail();
          break;
        }
        issue_w(s);
        issue_x(s);
        issued = s + 1;
      }
      if (*abort_flag) {
        // let the copies in flight land before shared memory goes away
        const int from = issued > p.sb ? issued - p.sb : 0;
        for (int s = from; s < issued; ++s)
          mbar_wait(full(s % p.sb), static_cast<uint32_t>(s / p.sb) & 1u, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------- consumers
    const int rb = warp % p.rbc, kp = warp / p.rbc;
    const int g = lane >> 2, t = lane & 3;
    const int ra = rb * 16 + g, rbw = ra + 8;           // the thread's two rows in the CTA
    // fp32 chains [group of the pair][half of the group]: with one token tile the
    // two halves of a group sum into separate accumulators (four independent MMA
    // chains: M <= 8 measured 16.05 -> 15.55 us at the decode shape); with more
    // tiles the registers go to the tiles (HS = 1)
    constexpr int HS = NT == 1 ? 2 : 1;
    float cf[2][HS][NT][4];
    int acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[j][i] = 0;
#pragma unroll
        for (int hh = 0; hh < HS; ++hh) cf[0][hh][j][i] = cf[1][hh][j][i] = 0.f;
      }
    int ng = 0;                                          // groups summed in cf (both)
    const ExpandMagic em = expand_magic();
    const uint32_t wpitch = static_cast<uint32_t>(p.gs) * 32;
    for (int s = 0; s < nslab; ++s) {
      const int b = s % p.sb;
      const bool got = mbar_wait(full(b), static_cast<uint32_t>(s / p.sb) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        fail();
        break;
      }
      int g0;
      const int n = slab_groups(s, &g0);
      const int lo = n * kp / p.kp, hi = n * (kp + 1) / p.kp;
      const uint8_t* buf = smem + b * p.buf_bytes;
      // two groups at a time into separate accumulators: two independent MMA chains
      for (int gl = lo; gl < hi; gl += 2) {
        const int npair = hi - gl >= 2 ? 2 : 1;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (u >= npair) break;
          const int gg = gl + u;
          const uint8_t* wra = buf + ra * wpitch + gg * 32 + t * 4;
          const uint8_t* wrb = buf + rbw * wpitch + gg * 32 + t * 4;
          const uint32_t wa[2] = {*reinterpret_cast<const uint32_t*>(wra),
                                  *reinterpret_cast<const uint32_t*>(wra + 16)};
          const uint32_t wb[2] = {*reinterpret_cast<const uint32_t*>(wrb),
                                  *reinterpret_cast<const uint32_t*>(wrb + 16)};
          // q in [-127, 127] as fp16 without a conversion: 0x6480 + q is the
          // fp16 of 1152 + q (exact), minus 1152
          const __half qa = __hsub(__ushort_as_half(static_cast<unsigned short>(
                                       0x6480 + static_cast<int8_t>(buf[p.off_q + gg * rows + ra]))),
                                   __ushort_as_half(0x6480));
          const __half qb = __hsub(__ushort_as_half(static_cast<unsigned short>(
                                       0x6480 + static_cast<int8_t>(buf[p.off_q + gg * rows + rbw]))),
                                   __ushort_as_half(0x6480));
          const __half2 qa2 = __halves2half2(qa, qa), qb2 = __halves2half2(qb, qb);
          const uint8_t* bcol = buf + p.off_b + (gg * kGroup + 16 * t) * 2;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // word t + 4h of the group: fp16 pairs (columns 16 (t + 4h) + 2e, + 1), e = 0..7
            uint32_t ea[8], eb[8];
            expand_word(wa[h], qa2, ea, em);
            expand_word(wb[h], qb2, eb, em);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const int tok = 8 * j + g;                 // B column g of n-tile j
              uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
              if (tok < M) {
                const uint8_t* bp = bcol + tok * p.b_pitch + h * 128;
                x0 = *reinterpret_cast<const uint4*>(bp);
                x1 = *reinterpret_cast<const uint4*>(bp + 16);
              }
              float (&c)[4] = cf[u][h % HS][j];
              mma_f16(c, ea[0], eb[0], ea[1], eb[1], x0.x, x0.y);
              mma_f16(c, ea[2], eb[2], ea[3], eb[3], x0.z, x0.w);
              mma_f16(c, ea[4], eb[4], ea[5], eb[5], x1.x, x1.y);
              mma_f16(c, ea[6], eb[6], ea[7], eb[7], x1.z, x1.w);
            }
          }
        }
        ng += npair;
        if (ng >= 2 * (kBlock / kGroup) - 1) {
          // each accumulator has summed at most eight groups: integers below 2^24
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int hh = 0; hh < HS; ++hh)
#pragma unroll
              for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  acc[j][i] += __float2int_rn(cf[u][hh][j][i]), cf[u][hh][j][i] = 0.f;
          ng = 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(b));
    }
    // C fragment: rows ra (i = 0, 1) and rbw (i = 2, 3), tokens 8j + 2t + (i & 1)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = 8 * j + 2 * t + (i & 1);
        int a = acc[j][i];
#pragma unroll
        for (int hh = 0; hh < HS; ++hh)
          a += __float2int_rn(cf[0][hh][j][i]) + __float2int_rn(cf[1][hh][j][i]);
        if (m < M) atomicAdd(red + ((i < 2) ? ra : rbw) * MP4 + m, a);
      }
    }
  }
  __syncwarp();
  __syncthreads();
  const bool ok = *abort_flag == 0;
  if (p.cs > 1) {
    if (crank != 0 && ok) {
      for (int i = threadIdx.x; i < rows * MP4; i += blockDim.x) {
        const int32_t v = red[i];
        if (v != 0) red_add_peer(peer_addr(red + i, 0), static_cast<uint32_t>(v));
      }
    }
    cluster_sync();
    if (crank != 0) return;
  }
  if (!ok) return;
  for (int i = threadIdx.x; i < rows * M; i += blockDim.x) {
    const int r = i % rows, m = i / rows;
    const int n = row0 + r;
    const int32_t a = red[r * MP4 + m];
    const size_t idx = static_cast<size_t>(m) * N + n;
    if (acc_dbg != nullptr) acc_dbg[idx] = a;
    store_y(y, y_dtype, idx, __fmul_rn(__fmul_rn(__int2float_rn(a), sw[n]), sx[m]));
  }
}

// The work split of a problem on `sms` SMs (see TcPlan).
TcPlan plan_tc(int M, int N, int K, int sms) {
  const int rowblocks = N / 16;
  const int G = K / kGroup;
  TcPlan p{};
  // the most rows per CTA (the activation image is read once per CTA) that
  // still gives about one CTA per SM, the cluster splitting K when needed
  int best_rbc = 1, best_cs = 1, best_ctas = 0;
  bool found = false;
  for (int rbc = 8; rbc >= 1 && !found; rbc >>= 1) {
    for (int cs = 1; cs <= 4 && cs <= G; cs <<= 1) {
      const int ctas = rowblocks / rbc * cs;
      if (ctas > best_ctas) {
        best_ctas = ctas;
        best_rbc = rbc;
        best_cs = cs;
      }
      if (10 * ctas >= 9 * sms) {
        best_rbc = rbc;
        best_cs = cs;
        best_ctas = ctas;
        found = true;
        break;
      }
    }
  }
  p.rbc = best_rbc;
  p.kp = kTcConsumers / best_rbc;
  p.cs = best_cs;
  const int rows = 16 * p.rbc;
  const int MP4 = (M + 3) & ~3;
  const int ggroups = (G + p.cs - 1) / p.cs;            // groups of the largest CTA range
  // two CTAs per SM when the grid exceeds the SMs
  const uint32_t budget = best_ctas > sms ? 100u * 1024 : 200u * 1024;
  const uint32_t red_bytes = static_cast<uint32_t>(rows) * MP4 * 4;
  const int gs_options[4] = {7, 5, 3, 1};
  for (int gs : gs_options) {
    if (gs > ggroups && gs != 1) continue;
    uint32_t off_q = rows * gs * 32;
    off_q = (off_q + 127) & ~127u;
    uint32_t off_b = off_q + rows * gs;
    off_b = (off_b + 127) & ~127u;
    // token rows of gs * 256 bytes at a pitch of 16 mod 128: conflict-free 16-byte reads
    const uint32_t pitch = static_cast<uint32_t>(gs) * 256 + 16;
    uint32_t buf = off_b + pitch * M;
    buf = (buf + 1023) & ~1023u;
    const uint32_t fixed = red_bytes + 16 * kTcMaxBuffers + 16;
    int sb = static_cast<int>((budget - fixed) / buf);
    if (sb > kTcMaxBuffers) sb = kTcMaxBuffers;
    const int slabs = (ggroups + gs - 1) / gs;
    if (sb > slabs) sb = slabs;
    if (sb < 1) continue;
    if (sb < 3 && sb < slabs && gs != 1) continue;    // prefer a deeper ring of smaller slabs
    p.gs = gs;
    p.sb = sb;
    p.buf_bytes = buf;
    p.off_q = off_q;
    p.off_b = off_b;
    p.b_pitch = pitch;
    p.red_off = static_cast<uint32_t>(sb) * buf;
    p.bar_off = (p.red_off + red_bytes + 15) & ~15u;
    p.smem = p.bar_off + 16 * sb + 16;
    return p;
  }
  p.gs = 0;   // nothing fits
  return p;
}

}  // namespace

cudaError_t launch_decode_tc(const uint8_t* packed, const int8_t* qT, const float* sw,
                             const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                             int y_dtype, int32_t* acc_dbg, int* status, cudaStream_t st) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const TcPlan p = plan_tc(M, N, K, sms);
  if (p.gs == 0) return cudaErrorInvalidConfiguration;
  const int rows = 16 * p.rbc;
  const int G = K / kGroup;
  CUtensorMap mw, mq;
  if (!make_map_2d(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, static_cast<uint64_t>(K) / 4, N,
                   static_cast<uint64_t>(K) / 4, p.gs * 32, rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qT, N, G, static_cast<uint64_t>(N), rows,
                   p.gs, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const size_t smem = p.smem + 1024;
  const int ctas = N / rows * p.cs;
  const int mt = (M + 7) / 8;   // n-tiles of 8 tokens
  auto go = [&](auto kernel) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (r != cudaSuccess) return r;
    return launch_pdl_cluster(kernel, dim3(ctas), dim3(kTcThreads), smem, st, p.cs, mw, mq, xq, sw,
                              sx, M, N, K, p, y, y_dtype, acc_dbg, status);
  };
  if (mt <= 1) return go(decode_tc_kernel<1>);
  if (mt <= 2) return go(decode_tc_kernel<2>);
  if (mt <= 3) return go(decode_tc_kernel<3>);
  return go(decode_tc_kernel<4>);
}

}  // namespace tl
