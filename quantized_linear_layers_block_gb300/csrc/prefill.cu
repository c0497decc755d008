// K3: prefill ternary linear layer on the 5th-generation tensor cores.
//
// Qiita item ecc183fae033565af7cb §4 "効いた高速化" turns the layer into one
// int8 GEMM plus a per-row and per-token rescale; §6 "部品ごとに測る" measured
// the separate int8 weight expansion at 31 of 83 ms. Here the expansion lives
// inside the GEMM's main loop and the expanded weights never touch memory.
//
// sm_103a has no integer tcgen05 MMA, so the int8 operands are fed to
// tcgen05.mma kind::f16 as fp16 (every int8 value is exact in fp16, every
// product |x w| <= 16129 is exact in fp32). One 1024-column chunk of K is
// accumulated in fp32 in tensor memory: each partial sum is an integer of
// magnitude <= 127*127*1024 = 16,516,096 < 2^24, so it is exact. The chunk
// results are then converted to int32 and summed exactly. The int32 result
// equals the int8 GEMM's bit for bit.
//
// Roles (one CTA per SM, persistent over output tiles of 128 weight rows x
// 128 tokens; the MMA is D[n, m] = sum_k W[n, k] X[m, k], i.e. y transposed):
//   warp 0      TMA producer: per 64-column stage, the fp16 activation tile
//               (128-byte swizzle), the packed 2-bit codes of the 128 rows and
//               their q bytes, into a 6-deep shared-memory ring.
//   warp 1      allocates tensor memory; one thread issues the MMAs.
//   warps 4-7   expansion: lane = weight row; decode 64 codes with q into 32
//               fp16 pairs in registers and store them into tensor memory as
//               the MMA's A operand (tcgen05.st), one 32-column slot per stage.
//   warps 8-15  drain + epilogue: after each chunk read the fp32 accumulator
//               (double buffered), add it to int32 totals in registers; at the
//               end of a tile write y = (fl32(acc) sw[n]) sx[m].
// Tensor memory (512 columns x 128 lanes): A slots at columns 32 s, the two
// fp32 accumulators at columns 256 and 384.
// When the problem has fewer tiles than SMs, K is split across CTAs; partial
// int32 sums meet in a caller workspace and the last CTA of a tile finishes it.
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace tl {
namespace {

constexpr int BM = 128;             // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;             // tokens per tile (MMA N)
constexpr int BK = 64;              // columns of K per pipeline stage
constexpr int NST = 6;              // pipeline depth
constexpr int STAGES_PER_CHUNK = kBlock / BK;
constexpr int UMMA_K = 16;

constexpr int B_BYTES = BN * BK * 2;          // 16 KB fp16 activation tile
constexpr int P_BYTES = BM * (BK / 4);        // 2 KB packed codes
constexpr int Q_BYTES = BM;                   // 128 q bytes
constexpr uint32_t STAGE_TX = B_BYTES + P_BYTES + Q_BYTES;

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = 0;                // A slot s at columns 32 s
constexpr uint32_t D_COL0 = 256;              // accumulators at 256 and 384

constexpr int kThreads = 512;
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_EXP0 = 4, WARP_DRAIN0 = 8;

constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

struct Smem {
  // byte offsets inside the 1024-aligned dynamic shared memory block
  static constexpr int b = 0;
  static constexpr int p = b + NST * B_BYTES;
  static constexpr int q = p + NST * P_BYTES;
  static constexpr int bar = q + NST * Q_BYTES;     // 8-byte aligned
  static constexpr int n_bars = 3 * NST + 2 + 2 + 3;
  static constexpr int misc = bar + n_bars * 8;
  static constexpr int total = misc + 16;
};

struct Work {
  int units, split, mtiles, chunks;
};

__device__ __forceinline__ void unit_coords(const Work& w, int u, int& nt, int& mt, int& c0,
                                            int& c1) {
  const int tile = u / w.split;
  const int sp = u % w.split;
  mt = tile % w.mtiles;
  nt = tile / w.mtiles;
  c0 = sp * w.chunks / w.split;
  c1 = (sp + 1) * w.chunks / w.split;
}

__device__ __forceinline__ void store_out(void* y, int y_dtype, size_t idx, float v) {
  if (y_dtype == TL_F32)
    static_cast<float*>(y)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// Expand one packed word (16 codes, layout of tl.h) into 8 fp16 pairs code*q.
// The 2-bit field e (= code + 1) is dropped into the mantissa of an fp16 whose
// exponent makes the value 2^E + e exactly; subtracting 2^E + 1 leaves the code
// in {-1, 0, +1} and one multiply by q gives code * q, all exact.
__device__ __forceinline__ void expand_word(uint32_t w, __half2 q2, uint32_t* out) {
  const __half2 c0 = __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401));  // 1025
  const __half2 c1 = __halves2half2(__ushort_as_half(0x5C04), __ushort_as_half(0x5C04));  // 257
  const __half2 c2 = __halves2half2(__ushort_as_half(0x5410), __ushort_as_half(0x5410));  // 65
  const __half2 c3 = __halves2half2(__ushort_as_half(0x4C40), __ushort_as_half(0x4C40));  // 17
  const __half2 c4 = __halves2half2(__ushort_as_half(0x4500), __ushort_as_half(0x4500));  // 5
  const __half2 cs[5] = {c0, c1, c2, c3, c4};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int jj = j < 5 ? j : j - 5;
    const uint32_t src = j < 5 ? w : (w >> 10);
    const uint32_t magic = static_cast<uint32_t>(25 - 2 * jj) << 10;
    const uint32_t bits = (src & (0x00030003u << (2 * jj))) | (magic | (magic << 16));
    __half2 h = *reinterpret_cast<const __half2*>(&bits);
    h = __hmul2(__hsub2(h, cs[jj]), q2);
    out[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_p,
               const __grid_constant__ CUtensorMap map_q, const float* __restrict__ sw,
               const float* __restrict__ sx, int M, int N, Work work, void* __restrict__ y,
               int y_dtype, int32_t* __restrict__ acc_dbg, int32_t* __restrict__ ws_acc,
               int* __restrict__ ws_cnt, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Smem::bar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (NST + s); };
  auto afull = [&](int s) { return bar0 + 8u * (2 * NST + s); };
  auto dfull = [&](int b) { return bar0 + 8u * (3 * NST + b); };
  auto dempty = [&](int b) { return bar0 + 8u * (3 * NST + 2 + b); };
  const uint32_t fin = bar0 + 8u * (3 * NST + 4);
  const uint32_t rdv1 = bar0 + 8u * (3 * NST + 5);
  const uint32_t rdv2 = bar0 + 8u * (3 * NST + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem::misc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + Smem::misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(afull(s), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(dfull(b), 1);
      mbar_init(dempty(b), 8);
    }
    mbar_init(fin, 1);
    mbar_init(rdv1, 8);
    mbar_init(rdv2, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(status, TL_ETIMEOUT);
  };

  if (warp == WARP_TMA) {
    if (lane == 0) {
      tma_prefetch_desc(&map_x);
      tma_prefetch_desc(&map_p);
      tma_prefetch_desc(&map_q);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < work.units; u += gridDim.x) {
        int nt, mt, c0, c1;
        unit_coords(work, u, nt, mt, c0, c1);
        for (int c = c0; ok && c < c1; ++c) {
          for (int st = 0; st < STAGES_PER_CHUNK; ++st, ++it) {
            const int s = it % NST;
            const uint32_t ph = (it / NST) & 1u;
            if (!mbar_wait(empty(s), ph ^ 1u, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            const int k0 = c * kBlock + st * BK;
            mbar_arrive_expect_tx(full(s), STAGE_TX);
            tma_load_2d(sbase + Smem::b + s * B_BYTES, &map_x, k0, mt * BN, full(s));
            tma_load_2d(sbase + Smem::p + s * P_BYTES, &map_p, k0 / 4, nt * BM, full(s));
            tma_load_2d(sbase + Smem::q + s * Q_BYTES, &map_q, nt * BM, k0 / kGroup, full(s));
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before shared memory goes away
        const uint32_t n = it < NST ? it : NST;
        for (uint32_t i = it - n; i < it; ++i) mbar_wait(full(i % NST), (i / NST) & 1u, nullptr);
      }
    }
  } else if (warp == WARP_MMA) {
    if (lane == 0) {
      uint32_t it = 0, cc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < work.units; u += gridDim.x) {
        int nt, mt, c0, c1;
        unit_coords(work, u, nt, mt, c0, c1);
        for (int c = c0; ok && c < c1; ++c, ++cc) {
          const uint32_t buf = cc & 1u;
          const uint32_t dph = (cc >> 1) & 1u;
          if (!mbar_wait(dempty(buf), dph ^ 1u, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_addr = tmem + D_COL0 + buf * BN;
          for (int st = 0; st < STAGES_PER_CHUNK; ++st, ++it) {
            const int s = it % NST;
            const uint32_t ph = (it / NST) & 1u;
            if (!mbar_wait(full(s), ph, abort_flag) || !mbar_wait(afull(s), ph, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t b_addr = sbase + Smem::b + s * B_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              mma_f16_ts(d_addr, tmem + A_COL0 + 32u * s + 8u * kk,
                         smem_desc_sw128(b_addr + 32u * kk), IDESC, (st | kk) != 0);
            }
            tc_commit(empty(s));
          }
          if (ok) tc_commit(dfull(buf));
        }
      }
      // all MMAs issued by this thread have finished before tensor memory is released
      tc_commit(fin);
      mbar_wait(fin, 0, nullptr);
    }
  } else if (warp >= WARP_EXP0 && warp < WARP_EXP0 + 4) {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < work.units; u += gridDim.x) {
      int nt, mt, c0, c1;
      unit_coords(work, u, nt, mt, c0, c1);
      for (int c = c0; ok && c < c1; ++c) {
        for (int st = 0; st < STAGES_PER_CHUNK; ++st, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1u;
          const bool got = mbar_wait(full(s), ph, abort_flag) && mbar_wait(empty(s), ph ^ 1u, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint4 pk = *reinterpret_cast<const uint4*>(smem + Smem::p + s * P_BYTES + row * 16);
          const int qv = static_cast<int8_t>(smem[Smem::q + s * Q_BYTES + row]);
          const __half qh = __int2half_rn(qv);
          const __half2 q2 = __halves2half2(qh, qh);
          uint32_t out[32];
          expand_word(pk.x, q2, out + 0);
          expand_word(pk.y, q2, out + 8);
          expand_word(pk.z, q2, out + 16);
          expand_word(pk.w, q2, out + 24);
          tmem_st_32x32b_x32(lane_base + A_COL0 + 32u * s, out);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull(s));
        }
      }
    }
  } else if (warp >= WARP_DRAIN0) {
    const int quarter = warp & 3;
    const int half = (warp - WARP_DRAIN0) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t cc = 0, ku = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < work.units; u += gridDim.x) {
      int nt, mt, c0, c1;
      unit_coords(work, u, nt, mt, c0, c1);
      int tot[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) tot[j] = 0;
      for (int c = c0; c < c1; ++c, ++cc) {
        const uint32_t buf = cc & 1u;
        const uint32_t dph = (cc >> 1) & 1u;
        const bool got = mbar_wait(dfull(buf), dph, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(lane_base + D_COL0 + buf * BN + half * 64 + p * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) tot[p * 32 + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty(buf));
      }
      const int n = nt * BM + row;
      const int mbase = mt * BN + half * 64;
      bool finish = ok;
      if (work.split > 1) {
        // Rendezvous of the 8 drain warps through two mbarriers (bounded waits):
        // every warp adds its partial sums, the leader counts the tile's
        // finished splits, and the CTA that completes the tile writes it.
        const uint32_t rp = ku & 1u;
        ++ku;
        if (ok) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int m = mbase + j;
            if (m < M) atomicAdd(ws_acc + static_cast<size_t>(m) * N + n, tot[j]);
          }
          __threadfence();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rdv1);
        if (warp == WARP_DRAIN0 && lane == 0) {
          int last = 0;
          if (mbar_wait(rdv1, rp, abort_flag)) {
            if (!*abort_flag) {
              __threadfence();
              last = atomicAdd(ws_cnt + u / work.split, 1) == work.split - 1;
            }
          } else {
            fail();
          }
          *last_flag = last;
          mbar_arrive(rdv2);
        }
        const bool got = mbar_wait(rdv2, rp, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          fail();
          ok = false;
        }
        finish = ok && *last_flag != 0;
        if (finish) {
          __threadfence();
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int m = mbase + j;
            if (m < M) tot[j] = __ldcg(ws_acc + static_cast<size_t>(m) * N + n);
          }
        }
      }
      if (finish) {
        const float swn = sw[n];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int m = mbase + j;
          if (m < M) {
            const size_t idx = static_cast<size_t>(m) * N + n;
            if (acc_dbg != nullptr) acc_dbg[idx] = tot[j];
            store_out(y, y_dtype, idx, __fmul_rn(__fmul_rn(__int2float_rn(tot[j]), swn), sx[m]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, CUtensorMapDataType dt,
                 const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int choose_split(int tiles, int chunks, int num_sms) {
  if (tiles >= num_sms) return 1;
  int s = (num_sms + tiles - 1) / tiles;
  return s < chunks ? s : chunks;
}

}  // namespace

size_t prefill_workspace_bytes(int M, int N, int K, int num_sms) {
  const int mtiles = (M + BN - 1) / BN;
  const int tiles = mtiles * (N / BM);
  if (choose_split(tiles, K / kBlock, num_sms) <= 1) return 0;
  return static_cast<size_t>(M) * N * 4 + static_cast<size_t>(tiles) * 4;
}

int launch_prefill(const PrefillArgs& a, int* status, cudaStream_t st, cudaError_t* cerr) {
  *cerr = cudaSuccess;
  auto enc = get_encode_fn();
  if (enc == nullptr) {
    *cerr = cudaErrorNotSupported;
    return TL_ECUDA;
  }
  int dev = 0, num_sms = 0;
  if ((*cerr = cudaGetDevice(&dev)) != cudaSuccess) return TL_ECUDA;
  if ((*cerr = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return TL_ECUDA;

  const int G = a.K / kGroup;
  CUtensorMap mx, mp, mq;
  if (!make_map_2d(enc, &mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.xq, a.K, a.M,
                   static_cast<uint64_t>(a.K) * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(enc, &mp, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, a.K / 4, a.N,
                   static_cast<uint64_t>(a.K) / 4, BK / 4, BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qT, a.N, G, static_cast<uint64_t>(a.N),
                   BM, 1, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return TL_EINVAL;
  }

  Work w;
  w.mtiles = (a.M + BN - 1) / BN;
  w.chunks = a.K / kBlock;
  const int tiles = w.mtiles * (a.N / BM);
  w.split = choose_split(tiles, w.chunks, num_sms);
  int32_t* ws_acc = nullptr;
  int* ws_cnt = nullptr;
  if (w.split > 1) {
    const size_t need = static_cast<size_t>(a.M) * a.N * 4 + static_cast<size_t>(tiles) * 4;
    if (a.workspace == nullptr || a.ws_bytes < need) {
      w.split = 1;
    } else {
      ws_acc = static_cast<int32_t*>(a.workspace);
      ws_cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) +
                                      static_cast<size_t>(a.M) * a.N * 4);
      if ((*cerr = cudaMemsetAsync(a.workspace, 0, need, st)) != cudaSuccess) return TL_ECUDA;
    }
  }
  w.units = tiles * w.split;
  const int grid = w.units < num_sms ? w.units : num_sms;
  const size_t smem = Smem::total + 1024;
  if ((*cerr = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem))) != cudaSuccess)
    return TL_ECUDA;
  prefill_kernel<<<grid, kThreads, smem, st>>>(mx, mp, mq, a.sw, a.sx, a.M, a.N, w, a.y,
                                               a.y_dtype, a.acc_dbg, ws_acc, ws_cnt, status);
  if ((*cerr = cudaGetLastError()) != cudaSuccess) return TL_ECUDA;
  return TL_OK;
}

}  // namespace tl

// ------------------------------------------------------------------ library-owned scratch
// Split-K scratch for tl_linear_prefill_noalloc: a fixed array that every
// device loading this library holds until the process exits. Host code must
// not pass the symbol itself to a kernel (on the host it is only a stand-in);
// the device address is looked up once per device below.
static __device__ __align__(256) unsigned char g_prefill_scratch[TL_NOALLOC_SCRATCH_BYTES];

namespace tl {

int prefill_noalloc_scratch(void** ptr) {
  static void* cache[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TL_ECUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr) return TL_ECUDA;
    cache[dev] = p;
  }
  *ptr = cache[dev];
  return TL_OK;
}

}  // namespace tl
