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
// Work: persistent CTAs (one per SM) over output tiles of 128 weight rows x
// BN tokens; the MMA computes D[n, m] = sum_k W[n, k] X[m, k] (y transposed,
// weight rows on the tensor-memory lanes), 256 columns of K per pipeline
// stage (16 MMAs of K = 16). BN is 128 for long batches and 64, 32 or 16
// (the MMA's N) when the batch has at most that many tokens: a weight tile is
// then expanded once for the whole batch while the tensor cores do no work on
// padding tokens, and the smaller activation tiles leave shared memory to a
// deeper weight ring, which the weight stream needs at these sizes.
// Roles of the warps (20 with two expansion warps per lane quarter, 28 with four):
//   warp 0       weight producer: packed 2-bit codes of the 128 rows and their
//                two q bytes per row and stage into a 4-deep ring (TMA); it
//                starts before the kernel waits for the preceding one
//                (programmatic dependent launch). Like warps 1 and 2, the whole
//                warp runs the loop and one elected lane issues.
//   warp 2       activation producer: after that wait, the fp16 activation tile
//                of the stage (four 128-byte-swizzled boxes of 64 columns) into a
//                3-deep ring.
//   warp 1       allocates tensor memory and issues the MMAs. The whole warp
//                runs the loop on warp-uniform values and one elected lane
//                issues: per stage it waits for the activation tile and the
//                A slot, issues the stage's 16 MMAs as one block of
//                straight-line code and commits the A slot and the activation
//                slot free. Every instruction on
//                this path delays the tensor pipe (the warp shares its SM
//                sub-partition with busy warps), so it does nothing else; the
//                warp-uniform form measured 146 -> 135.5 us at the gate+up
//                shape with 512 tokens against one lane running the loop.
//   expansion    EPQ (2 or 4) warps per 32-lane quarter of tensor memory: lane
//                = weight row; warp `part` turns its 256 / EPQ codes of the
//                stage (q group part / (EPQ / 2)) into fp16 pairs in registers
//                and stores them into tensor memory as the MMA's A operand
//                (tcgen05.st), then arrives on the A slot's full barrier (the
//                activations are the MMA warp's wait: a wait taken out of the
//                expansion warps' per-stage chain measured 133.8 -> 124.9 us
//                at the gate+up shape with 512 tokens).
//   drain        two warps per quarter (BN / 2 tokens each): after each
//                1024-column chunk add the fp32 accumulator (double buffered)
//                into int32 totals in registers; at the end of a tile write
//                y = (fl32(acc) sw[n]) sx[m].
// Tensor memory (512 columns x 128 lanes): NA A slots of 128 columns from
// column 0, then two fp32 accumulators of BN columns.
// When whole tiles would load the SMs unevenly (few tiles with a long K), the
// tiles of the last partial round are cut along K across CTAs; each piece
// stores its partial int32 sums in its own region of a caller workspace and
// the last CTA of a tile to arrive adds the others' regions, finishes it and
// returns the regions to zero, so the workspace needs zeroing only once, when
// it is allocated.
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace tl {
namespace {

constexpr int BM = 128;             // weight rows per tile (MMA M, TMEM lanes)
constexpr int BK = 256;             // columns of K per pipeline stage (two q groups)
constexpr int BOX_K = 64;           // columns per 128-byte swizzled activation box
constexpr int STAGES_PER_CHUNK = kBlock / BK;
constexpr int UMMA_K = 16;
constexpr int MMAS_PER_STAGE = BK / UMMA_K;
static_assert(MMAS_PER_STAGE == 16, "mma_stage16 issues one stage");
constexpr int P_BYTES = BM * (BK / 4);        // 8 KB packed codes
static_assert(BK / 4 == 64, "one 64-byte swizzle span of codes per weight row and stage");
constexpr int Q_BYTES = BM * (BK / kGroup);   // 256 q bytes: [2 groups][128 rows]
constexpr uint32_t W_TX = P_BYTES + Q_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COLS = BK / 2;           // 128 columns of fp16 pairs per A slot
constexpr int WARP_WLOAD = 0, WARP_MMA = 1, WARP_BLOAD = 2, WARP_EXP0 = 4;
constexpr int N_DRAIN_WARPS = 8;

// Per tile width BN (tokens): ring depths (NW weight stages, NB activation
// stages, NA tensor-memory A slots) and expansion warps per lane quarter (EPQ).
template <int BN_, int NW_, int NB_, int NA_, int EPQ_>
struct Cfg {
  static constexpr int BN = BN_, NW = NW_, NB = NB_, NA = NA_, EPQ = EPQ_;
  static constexpr int BOX_BYTES = BN * BOX_K * 2;   // one 128-byte swizzled box
  static constexpr int B_BYTES = BN * BK * 2;        // fp16 activation tile of a stage (four boxes)
  static constexpr int N_EXP_WARPS = 4 * EPQ;
  static constexpr int WARP_DRAIN0 = WARP_EXP0 + N_EXP_WARPS;
  static constexpr int kThreads = (WARP_DRAIN0 + N_DRAIN_WARPS) * 32;
  static constexpr int EXP_COLS = A_COLS / EPQ;      // tensor-memory columns per expansion warp
  static constexpr int EXP_WORDS = EXP_COLS / 8;     // packed 16-code words per lane and stage
  static constexpr uint32_t D_COL0 = NA * A_COLS;    // accumulators at D_COL0 + {0, BN}
  static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
  // byte offsets inside the 1024-aligned dynamic shared memory block
  static constexpr int sb = 0;
  static constexpr int sp = sb + NB * B_BYTES;
  static constexpr int sq = sp + NW * P_BYTES;
  static constexpr int sbar = sq + NW * Q_BYTES;
  // wfull[NW] wempty[NW] bfull[NB] bempty[NB] afull[NA] aempty[NA] dfull[2] dempty[2] fin
  static constexpr int n_bars = 2 * NW + 2 * NB + 2 * NA + 2 + 2 + 1;
  static constexpr int smisc = sbar + n_bars * 8;
  static constexpr int stotal = smisc + 16;
  static_assert(stotal + 1024 <= 232448, "shared memory budget");
  static_assert(D_COL0 + 2 * BN <= TMEM_COLS, "tensor memory budget");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(EPQ == 2 || EPQ == 4, "expansion split");
};
// 128 tokens: the activation ring fills shared memory; 64, 32 and 16 tokens:
// deeper weight rings and a third A slot; four expansion warps per quarter
// where the drain's totals are few enough for the smaller register budget.
using Cfg128 = Cfg<128, 4, 3, 2, 2>;
using Cfg64 = Cfg<64, 8, 4, 3, 2>;
using Cfg32 = Cfg<32, 12, 4, 3, 4>;
using Cfg16 = Cfg<16, 16, 4, 3, 4>;

// Work schedule. Tiles [0, full) are whole units, dealt round-robin to the
// grid (all of them unless plan_work finds the imbalance worth a cut). The
// remaining `tail` tiles form a chunk space of tail * chunks chunks that is
// cut into `tgrid` contiguous, equal ranges, one per CTA 0 .. tgrid-1 (each
// at least one chunk): a CTA's range covers pieces of one or more tiles. A
// tile cut between CTAs meets in workspace slot (tile - full), through nreg
// regions: with few CTAs per tile (nreg = their most) every piece stores its
// int32 partial sums in its own region (contributor ci); with more (nreg = 1)
// every piece adds them into the one region with atomics. Per drain warp a
// counter tells the last of the tile's contributors to arrive, which gathers
// the sums and writes the tile.
struct Work {
  int mtiles, chunks, full, tail, tgrid, nreg;
};

struct Piece {
  int nt, mt, c0, c1;   // tile (weight-row block, token block) and chunk range
  int slot;             // workspace slot, or -1 for a whole tile
  int contrib;          // CTAs that share the tile (1 for a whole tile)
  int ci;               // this CTA's place among them
};

__device__ __forceinline__ int num_pieces(const Work& w, int b) {
  const int grid = static_cast<int>(gridDim.x);
  int n = w.full > b ? (w.full - b - 1) / grid + 1 : 0;
  if (b < w.tgrid) {
    const int T = w.tail * w.chunks;
    const int s = b * T / w.tgrid, e = (b + 1) * T / w.tgrid;
    n += (e - 1) / w.chunks - s / w.chunks + 1;
  }
  return n;
}

__device__ __forceinline__ Piece get_piece(const Work& w, int b, int k) {
  const int grid = static_cast<int>(gridDim.x);
  const int nfull = w.full > b ? (w.full - b - 1) / grid + 1 : 0;
  Piece p;
  int tile;
  if (k < nfull) {
    tile = b + k * grid;
    p.c0 = 0;
    p.c1 = w.chunks;
    p.slot = -1;
    p.contrib = 1;
    p.ci = 0;
  } else {
    const int T = w.tail * w.chunks;
    const int s = b * T / w.tgrid, e = (b + 1) * T / w.tgrid;
    const int tt = s / w.chunks + (k - nfull);          // tile within the tail
    const int lo = tt * w.chunks, hi = lo + w.chunks;
    p.c0 = (s > lo ? s : lo) - lo;
    p.c1 = (e < hi ? e : hi) - lo;
    // owner of chunk i: the CTA c with c T / tgrid <= i < (c + 1) T / tgrid
    const int first = ((lo + 1) * w.tgrid - 1) / T;
    const int last = (hi * w.tgrid - 1) / T;
    p.contrib = last - first + 1;
    p.ci = b - first;
    p.slot = p.contrib > 1 ? tt : -1;
    tile = w.full + tt;
  }
  p.mt = tile % w.mtiles;
  p.nt = tile / w.mtiles;
  return p;
}

__device__ __forceinline__ void store_out(void* y, int y_dtype, size_t idx, float v) {
  if (y_dtype == TL_F32)
    static_cast<float*>(y)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "r"(taddr)
      : "memory");
}

// Adds the fp32 accumulator columns [col, col + W) of this warp's lanes,
// integers below 2^24 in magnitude, to the int32 totals.
template <int W>
__device__ __forceinline__ void drain_add(uint32_t taddr, int (&tot)[W]) {
  if constexpr (W == 8) {
    uint32_t v[8];
    tmem_ld_32x32b_x8(taddr, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 8; ++i) tot[i] += __float2int_rn(__uint_as_float(v[i]));
  } else {
#pragma unroll
    for (int p = 0; p < W / 16; ++p) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(taddr + p * 16, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) tot[p * 16 + i] += __float2int_rn(__uint_as_float(v[i]));
    }
  }
}


// The 16 MMAs of a stage: A columns a + 8 j, B boxes j / 4 (low descriptor
// words b0..b3, high word bhi) at K steps j % 4 (32 bytes = 2 units each);
// the first accumulates only if acc != 0.
__device__ __forceinline__ void mma_stage16(uint32_t d, uint32_t a, uint32_t b0, uint32_t b1,
                                            uint32_t b2, uint32_t b3, uint32_t bhi, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p0, p1;\n .reg .b32 t;\n .reg .b64 bd;\n"
      "setp.ne.b32 p0, %8, 0;\n setp.eq.b32 p1, %8, %8;\n"
      "mov.b64 bd, {%2, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %7, p0;\n"
      "add.u32 t, %2, 2;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+8], bd, %7, p1;\n"
      "add.u32 t, %2, 4;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+16], bd, %7, p1;\n"
      "add.u32 t, %2, 6;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+24], bd, %7, p1;\n"
      "mov.b64 bd, {%3, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+32], bd, %7, p1;\n"
      "add.u32 t, %3, 2;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+40], bd, %7, p1;\n"
      "add.u32 t, %3, 4;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+48], bd, %7, p1;\n"
      "add.u32 t, %3, 6;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+56], bd, %7, p1;\n"
      "mov.b64 bd, {%4, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+64], bd, %7, p1;\n"
      "add.u32 t, %4, 2;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+72], bd, %7, p1;\n"
      "add.u32 t, %4, 4;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+80], bd, %7, p1;\n"
      "add.u32 t, %4, 6;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+88], bd, %7, p1;\n"
      "mov.b64 bd, {%5, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+96], bd, %7, p1;\n"
      "add.u32 t, %5, 2;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+104], bd, %7, p1;\n"
      "add.u32 t, %5, 4;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+112], bd, %7, p1;\n"
      "add.u32 t, %5, 6;\n mov.b64 bd, {t, %6};\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+120], bd, %7, p1;\n"
      "}" ::"r"(d), "r"(a), "r"(b0), "r"(b1), "r"(b2), "r"(b3), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}

// Two commits: both barriers see one arrival when the MMAs issued so far complete.
__device__ __forceinline__ void tc_commit2(uint32_t bar1, uint32_t bar2) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];" ::"r"(bar1),
      "r"(bar2)
      : "memory");
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_p,
               const __grid_constant__ CUtensorMap map_q, const float* __restrict__ sw,
               const float* __restrict__ sx, int M, int N, Work work, void* __restrict__ y,
               int y_dtype, int32_t* __restrict__ acc_dbg, int32_t* __restrict__ ws_acc,
               int* __restrict__ ws_cnt, int* status) {
  constexpr int BN = C::BN, NW = C::NW, NB = C::NB, NA = C::NA;
  constexpr int N_EXP_WARPS = C::N_EXP_WARPS, WARP_DRAIN0 = C::WARP_DRAIN0;
  constexpr int HB = BN / 2;                 // tokens per drain warp
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned (through an integer: the generic loads this gives the
  // expansion warps measured faster here than shared-space ones, 153 against
  // 160 us at the gate+up shape with 512 tokens)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::sbar;
  auto wfull = [&](int i) { return bar0 + 8u * i; };
  auto wempty = [&](int i) { return bar0 + 8u * (NW + i); };
  auto bfull = [&](int i) { return bar0 + 8u * (2 * NW + i); };
  auto bempty = [&](int i) { return bar0 + 8u * (2 * NW + NB + i); };
  auto afull = [&](int i) { return bar0 + 8u * (2 * NW + 2 * NB + i); };
  auto aempty = [&](int i) { return bar0 + 8u * (2 * NW + 2 * NB + NA + i); };
  auto dfull = [&](int i) { return bar0 + 8u * (2 * NW + 2 * NB + 2 * NA + i); };
  auto dempty = [&](int i) { return bar0 + 8u * (2 * NW + 2 * NB + 2 * NA + 2 + i); };
  const uint32_t fin = bar0 + 8u * (2 * NW + 2 * NB + 2 * NA + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::smisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::smisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(wfull(i), 1);
      mbar_init(wempty(i), N_EXP_WARPS);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(bfull(i), 1);
      mbar_init(bempty(i), 1);
    }
    for (int i = 0; i < NA; ++i) {
      // a stage is ready for the MMAs when all expansion warps have written
      // their part of its A slot and have seen its activation tile land
      mbar_init(afull(i), N_EXP_WARPS);
      mbar_init(aempty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(dfull(i), 1);
      mbar_init(dempty(i), N_DRAIN_WARPS);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
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

  // The single-thread roles (the two TMA producers and the MMA issuer) run
  // their loops on the whole warp with warp-uniform values; one elected lane
  // issues the copies, MMAs and commits.
  uint32_t elected;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(elected));
  if (warp == WARP_WLOAD) {
    {
      if (elected) {
        tma_prefetch_desc(&map_p);
        tma_prefetch_desc(&map_q);
      }
      uint32_t it = 0;
      bool ok = true;
      const int npieces = num_pieces(work, blockIdx.x);
      for (int k = 0; ok && k < npieces; ++k) {
        const Piece pc = get_piece(work, blockIdx.x, k);
        const int nt = pc.nt, c0 = pc.c0, c1 = pc.c1;
        for (int c = c0; ok && c < c1; ++c) {
          for (int st = 0; st < STAGES_PER_CHUNK; ++st, ++it) {
            const int w = it % NW;
            const uint32_t ph = (it / NW) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(wempty(w), ph ^ 1u, abort_flag))) {
              fail();
              ok = false;
              break;
            }
            const int k0 = c * kBlock + st * BK;
            if (elected) {
              mbar_arrive_expect_tx(wfull(w), W_TX);
              tma_load_2d(sbase + C::sp + w * P_BYTES, &map_p, k0 / 4, nt * BM, wfull(w));
              tma_load_2d(sbase + C::sq + w * Q_BYTES, &map_q, nt * BM, k0 / kGroup, wfull(w));
            }
            __syncwarp();
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before shared memory goes away
        const uint32_t n = it < NW ? it : NW;
        for (uint32_t i = it - n; i < it; ++i) mbar_wait(wfull(i % NW), (i / NW) & 1u, nullptr);
      }
    }
  } else if (warp == WARP_BLOAD) {
    {
      if (elected) tma_prefetch_desc(&map_x);
      // the activations are written by the preceding kernel in the stream
      pdl_wait_prior();
      uint32_t it = 0;
      bool ok = true;
      const int npieces = num_pieces(work, blockIdx.x);
      for (int k = 0; ok && k < npieces; ++k) {
        const Piece pc = get_piece(work, blockIdx.x, k);
        const int mt = pc.mt, c0 = pc.c0, c1 = pc.c1;
        for (int c = c0; ok && c < c1; ++c) {
          for (int st = 0; st < STAGES_PER_CHUNK; ++st, ++it) {
            const int b = it % NB;
            const uint32_t ph = (it / NB) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(bempty(b), ph ^ 1u, abort_flag))) {
              fail();
              ok = false;
              break;
            }
            const int k0 = c * kBlock + st * BK;
            if (elected) {
              mbar_arrive_expect_tx(bfull(b), C::B_BYTES);
#pragma unroll
              for (int bx = 0; bx < BK / BOX_K; ++bx)
                tma_load_2d(sbase + C::sb + b * C::B_BYTES + bx * C::BOX_BYTES, &map_x,
                            k0 + bx * BOX_K, mt * BN, bfull(b));
            }
            __syncwarp();
          }
        }
      }
      if (elected) pdl_launch_dependents();
      if (!ok) {
        const uint32_t n = it < NB ? it : NB;
        for (uint32_t i = it - n; i < it; ++i) mbar_wait(bfull(i % NB), (i / NB) & 1u, nullptr);
      }
    }
  } else if (warp == WARP_MMA) {
    {
      uint32_t cc = 0, aph = 0, bph = 0;
      int a = 0, b = 0;   // A slot and activation slot of the next stage
      bool ok = true;
      const uint64_t desc0 = smem_desc_sw128(sbase + C::sb);
      const uint32_t blo0 = static_cast<uint32_t>(desc0), bhi = static_cast<uint32_t>(desc0 >> 32);
      constexpr uint32_t BU = C::BOX_BYTES >> 4, SU = C::B_BYTES >> 4;
      const int npieces = num_pieces(work, blockIdx.x);
      for (int k = 0; ok && k < npieces; ++k) {
        const Piece pc = get_piece(work, blockIdx.x, k);
        const int c0 = pc.c0, c1 = pc.c1;
        for (int c = c0; ok && c < c1; ++c, ++cc) {
          const uint32_t buf = cc & 1u;
          const uint32_t dph = (cc >> 1) & 1u;
          if (!__all_sync(0xffffffffu, mbar_wait(dempty(buf), dph ^ 1u, abort_flag))) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_addr = tmem + C::D_COL0 + buf * BN;
#pragma unroll
          for (int st = 0; st < STAGES_PER_CHUNK; ++st) {
            if (!__all_sync(0xffffffffu, mbar_wait(bfull(b), bph, abort_flag) &&
                                             mbar_wait(afull(a), aph, abort_flag))) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t blo = blo0 + SU * b;
            if (elected) {
              mma_stage16(d_addr, tmem + A_COLS * a, blo, blo + BU, blo + 2 * BU, blo + 3 * BU, bhi,
                          C::IDESC, st != 0);
              tc_commit2(aempty(a), bempty(b));
            }
            __syncwarp();
            if (++a == NA) {
              a = 0;
              aph ^= 1u;
            }
            if (++b == NB) {
              b = 0;
              bph ^= 1u;
            }
          }
          if (ok && elected) tc_commit(dfull(buf));
          __syncwarp();
        }
      }
      if (elected) tc_commit(fin);
      __syncwarp();
      mbar_wait(fin, 0, nullptr);
    }
  } else if (warp >= WARP_EXP0 && warp < WARP_EXP0 + N_EXP_WARPS) {
    // EPQ warps per lane quarter; warp `part` expands tensor-memory columns
    // [EXP_COLS part, EXP_COLS (part + 1)) of every stage's A slot: the codes
    // 16 EXP_WORDS part .. of its row in the stage, all of one q group
    const int quarter = warp & 3;
    const int part = (warp - WARP_EXP0) >> 2;
    const int grp = part / (C::EPQ / 2);
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const ExpandMagic em = expand_magic();
    int w = 0, a = 0;            // weight and A slots of the stage
    uint32_t wph = 0, aph = 0;   // and their phases
    bool ok = true;
    const int npieces = num_pieces(work, blockIdx.x);
    for (int k = 0; ok && k < npieces; ++k) {
      const Piece pc = get_piece(work, blockIdx.x, k);
      const int c0 = pc.c0, c1 = pc.c1;
      for (int c = c0; ok && c < c1; ++c) {
        for (int st = 0; st < STAGES_PER_CHUNK; ++st) {
          const bool got = mbar_wait(wfull(w), wph, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            fail();
            ok = false;
            break;
          }
          // the codes arrive 64-byte swizzled (TMA): 16-byte chunk c of row r sits
          // at chunk c ^ ((r >> 1) & 3), so a quarter warp's eight rows hit all
          // eight bank groups (unswizzled rows 64 bytes apart conflict 4-way)
          const uint8_t* prow = smem + C::sp + w * P_BYTES + row * (BK / 4);
          uint4 pk[C::EXP_WORDS / 4];
#pragma unroll
          for (int i = 0; i < C::EXP_WORDS / 4; ++i) {
            const int chunk = part * (C::EXP_WORDS / 4) + i;
            pk[i] = *reinterpret_cast<const uint4*>(prow + ((chunk ^ ((row >> 1) & 3)) << 4));
          }
          const int qv = static_cast<int8_t>(smem[C::sq + w * Q_BYTES + grp * BM + row]);
          // the slot is refilled by TMA (async proxy): order these ordinary
          // loads before the release, or the copy can overtake them
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(wempty(w));   // weight slot consumed
          // q in [-127, 127] as fp16 without a conversion: 0x6400 + q + 128 is
          // the fp16 of 1152 + q, exact; subtracting 1152 leaves q
          const __half qh = __hsub(__ushort_as_half(static_cast<unsigned short>(0x6480 + qv)),
                                   __ushort_as_half(0x6480));
          const __half2 q2 = __halves2half2(qh, qh);
          uint32_t out[32];
          expand_word(pk[0].x, q2, out + 0, em);
          expand_word(pk[0].y, q2, out + 8, em);
          expand_word(pk[0].z, q2, out + 16, em);
          expand_word(pk[0].w, q2, out + 24, em);
          // the A slot is free once the MMAs of the stage that used it last completed
          const bool free_slot = mbar_wait(aempty(a), aph ^ 1u, abort_flag);
          if (!__all_sync(0xffffffffu, free_slot)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aslot = lane_base + A_COLS * a + C::EXP_COLS * part;
          tmem_st_32x32b_x32(aslot, out);
          if constexpr (C::EXP_WORDS == 8) {
            expand_word(pk[1].x, q2, out + 0, em);
            expand_word(pk[1].y, q2, out + 8, em);
            expand_word(pk[1].z, q2, out + 16, em);
            expand_word(pk[1].w, q2, out + 24, em);
            tmem_st_32x32b_x32(aslot + 32, out);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull(a));
          if (++w == NW) {
            w = 0;
            wph ^= 1u;
          }
          if (++a == NA) {
            a = 0;
            aph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= WARP_DRAIN0) {
    const int quarter = warp & 3;
    const int half = (warp - WARP_DRAIN0) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t cc = 0;
    bool ok = true;
    const int npieces = num_pieces(work, blockIdx.x);
    for (int k = 0; ok && k < npieces; ++k) {
      const Piece pc = get_piece(work, blockIdx.x, k);
      const int nt = pc.nt, mt = pc.mt, c0 = pc.c0, c1 = pc.c1;
      const int slot = pc.slot;
      int tot[HB];
#pragma unroll
      for (int j = 0; j < HB; ++j) tot[j] = 0;
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
        drain_add<HB>(lane_base + C::D_COL0 + buf * BN + half * HB, tot);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty(buf));
      }
      const int n = nt * BM + row;
      const int mbase = mt * BN + half * HB;
      bool finish = ok;
      if (slot >= 0 && ok) {
        // the warp's slice of the tile ([token][row] within a region): with one
        // region per contributor it stores its sums in its own (plain stores),
        // else it adds them into the single region; the warp's counter for the
        // tile then says whether every other contributor's same warp is done.
        // The last one gathers the sums, writes the tile and returns the
        // regions and the counter to zero for the next call.
        const size_t region = static_cast<size_t>(BM) * BN;
        int32_t* ws_tile = ws_acc + static_cast<size_t>(slot) * work.nreg * region + (half * HB) * BM + row;
        const bool own_regions = work.nreg > 1;
        int32_t* dst = ws_tile + (own_regions ? static_cast<size_t>(pc.ci) * region : 0);
#pragma unroll
        for (int j = 0; j < HB; ++j) {
          if (own_regions)
            __stcg(dst + j * BM, tot[j]);
          else
            atomicAdd(dst + j * BM, tot[j]);
        }
        __threadfence();
        __syncwarp();
        int* cnt = ws_cnt + slot * N_DRAIN_WARPS + (warp - WARP_DRAIN0);
        int last = 0;
        if (lane == 0) {
          last = atomicAdd(cnt, 1) == pc.contrib - 1;
          // every contributor has counted itself: nothing reads the count again
          if (last) *cnt = 0;
        }
        finish = __shfl_sync(0xffffffffu, last, 0) != 0;
        if (finish) {
          __threadfence();
          // own regions: add the others' (this CTA's sums are in tot already);
          // one shared region: it holds every piece's sums
          const int nparts = own_regions ? pc.contrib : 1;
#pragma unroll 1
          for (int c = 0; c < nparts; ++c) {
            int32_t* part = ws_tile + static_cast<size_t>(c) * region;
            const bool mine = own_regions && c == pc.ci;
#pragma unroll
            for (int j = 0; j < HB; ++j) {
              if (!mine) {
                const int v = __ldcg(part + j * BM);
                tot[j] = own_regions ? tot[j] + v : v;
              }
              __stcg(part + j * BM, 0);
            }
          }
        }
      } else if (slot >= 0) {
        finish = false;
      }
      if (finish) {
        const float swn = sw[n];
#pragma unroll
        for (int j = 0; j < HB; ++j) {
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
  // lanes of a warp can arrive here at different times (work done by one lane):
  // the warp converges first so that the CTA barrier below waits for every
  // thread (the tensor memory is released only after the last drain has read it)
  __syncwarp();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

// Tokens per tile for a batch of M tokens: the narrowest MMA N that holds the
// batch up to 64 tokens, 128 above.
int tile_tokens(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }

// The schedule of a problem (see Work) on `grid` CTAs, and the workspace
// bytes its split tiles need (0 when no tile is split).
size_t plan_work(int M, int N, int K, int num_sms, Work* w, int* grid) {
  const int bn = tile_tokens(M);
  w->mtiles = (M + bn - 1) / bn;
  w->chunks = K / kBlock;
  w->nreg = 1;
  const int tiles = w->mtiles * (N / BM);
  // whole tiles dealt round-robin, unless that leaves the busiest CTA more
  // than kSplitGain chunks above an even share: the meeting of a cut tile's
  // partial sums costs about that much (measured 14-18 us, 5-6 chunks), so a
  // smaller imbalance is cheaper to keep (17408 x 5120 with 256 tokens, 1.79
  // tiles per SM: 35.2 us whole against 41.0 cut; with 64 tokens, 0.89 tiles
  // per SM: 17.0 against 22.5; down_proj with 256 tokens, 80 tiles of 17
  // chunks: 41.7 cut against 52.7 whole)
  constexpr int kSplitGain = 6;
  *grid = tiles < num_sms ? tiles : num_sms;
  const int busiest = (tiles + num_sms - 1) / num_sms * w->chunks;
  const bool cut = static_cast<long long>(busiest) * num_sms - static_cast<long long>(tiles) * w->chunks >
                   static_cast<long long>(kSplitGain) * num_sms;
  if (!cut) {
    w->full = tiles;
    w->tail = 0;
    w->tgrid = 0;
    return 0;
  }
  // the tiles of the last partial round (all of them when there are fewer
  // tiles than SMs) are cut into equal chunk ranges over the CTAs; a tile
  // shared by at most three CTAs meets through one region per CTA (the
  // finishing CTA adds up to two regions), one shared by more through
  // atomics into one region (down_proj with 256 tokens, 80 tiles cut over 152
  // CTAs: 41.7 us through regions against 51.1 through atomics; 5120 x 17408
  // with 1024 tokens, 16 tiles cut over 152 CTAs: 116 us through atomics,
  // 132 through regions)
  *grid = num_sms;
  w->full = tiles / num_sms * num_sms;
  w->tail = tiles - w->full;
  const int T = w->tail * w->chunks;
  w->tgrid = T < num_sms ? T : num_sms;
  int maxc = 1;
  for (int tt = 0; tt < w->tail; ++tt) {   // the CTAs that share each tile (as get_piece)
    const int lo = tt * w->chunks, hi = lo + w->chunks;
    const int first = ((lo + 1) * w->tgrid - 1) / T, last = (hi * w->tgrid - 1) / T;
    if (last - first + 1 > maxc) maxc = last - first + 1;
  }
  w->nreg = maxc <= 3 ? maxc : 1;
  return static_cast<size_t>(w->tail) * w->nreg * (BM * bn) * 4 +
         static_cast<size_t>(w->tail) * N_DRAIN_WARPS * 4;
}

template <class C>
int launch_cfg(const PrefillArgs& a, int num_sms, int* status, cudaStream_t st, cudaError_t* cerr) {
  auto enc = get_encode_fn();
  if (enc == nullptr) {
    *cerr = cudaErrorNotSupported;
    return TL_ECUDA;
  }
  const int G = a.K / kGroup;
  CUtensorMap mx, mp, mq;
  if (!make_map_2d(enc, &mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.xq, a.K, a.M,
                   static_cast<uint64_t>(a.K) * 2, BOX_K, C::BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(enc, &mp, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, a.K / 4, a.N,
                   static_cast<uint64_t>(a.K) / 4, BK / 4, BM, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qT, a.N, G, static_cast<uint64_t>(a.N),
                   BM, BK / kGroup, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return TL_EINVAL;
  }

  Work w;
  int grid = 0;
  const size_t need = plan_work(a.M, a.N, a.K, num_sms, &w, &grid);
  int32_t* ws_acc = nullptr;
  int* ws_cnt = nullptr;
  if (need > 0) {
    if (a.workspace == nullptr || a.ws_bytes < need) {
      // no room: every tile whole, dealt round-robin
      w.full = w.mtiles * (a.N / BM);
      w.tail = 0;
      w.tgrid = 0;
      w.nreg = 1;
      if (grid > w.full) grid = w.full;
    } else {
      // the workspace is zero (zeroed by the caller once, and returned to zero
      // by every call that completes); the no-alloc entry clears it anyway
      ws_acc = static_cast<int32_t*>(a.workspace);
      ws_cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) +
                                      static_cast<size_t>(w.tail) * w.nreg * (BM * C::BN) * 4);
      if (a.clear_workspace &&
          (*cerr = cudaMemsetAsync(a.workspace, 0, need, st)) != cudaSuccess)
        return TL_ECUDA;
    }
  }
  const size_t smem = C::stotal + 1024;
  if ((*cerr = cudaFuncSetAttribute(prefill_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem))) != cudaSuccess)
    return TL_ECUDA;
  if ((*cerr = launch_pdl(prefill_kernel<C>, dim3(grid), dim3(C::kThreads), smem, st, mx, mp, mq,
                          a.sw, a.sx, a.M, a.N, w, a.y, a.y_dtype, a.acc_dbg, ws_acc, ws_cnt,
                          status)) != cudaSuccess)
    return TL_ECUDA;
  return TL_OK;
}

}  // namespace

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

size_t prefill_workspace_bytes(int M, int N, int K, int num_sms) {
  Work w;
  int grid = 0;
  return plan_work(M, N, K, num_sms, &w, &grid);
}

bool prefill_split_required(int M, int N, int num_sms) {
  const int bn = tile_tokens(M);
  return ((M + bn - 1) / bn) * (N / BM) < num_sms;
}

int launch_prefill(const PrefillArgs& a, int* status, cudaStream_t st, cudaError_t* cerr) {
  *cerr = cudaSuccess;
  int dev = 0, num_sms = 0;
  if ((*cerr = cudaGetDevice(&dev)) != cudaSuccess) return TL_ECUDA;
  if ((*cerr = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return TL_ECUDA;
  switch (tile_tokens(a.M)) {
    case 16: return launch_cfg<Cfg16>(a, num_sms, status, st, cerr);
    case 32: return launch_cfg<Cfg32>(a, num_sms, status, st, cerr);
    case 64: return launch_cfg<Cfg64>(a, num_sms, status, st, cerr);
    default: return launch_cfg<Cfg128>(a, num_sms, status, st, cerr);
  }
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
