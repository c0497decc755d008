/*
 * tl.h — C ABI of the GB300 (sm_103a) ternary linear layer library.
 *
 * The layer (Qiita item ecc183fae033565af7cb, "Ternary-Bonsai-2-27B on
 * 2x RTX 5070 12GB with vLLM TP=2", sections 前提 and §4 "効いた高速化"):
 *
 *   weights   code[n,k] in {-1,0,+1}, one fp16 scale s[n,g] per 128 columns
 *   rotation  xr = (1/32) H1024 x per 1024-column block (Sylvester order)
 *   weights   smax[n] = max_g |s[n,g]|, q[n,g] = rne(127 s[n,g] / smax[n]),
 *             W_int8[n,k] = code[n,k] q[n,k/128]  (|W_int8| <= 127)
 *   tokens    a = max_k |xr[m,k]|, xq = rne(xr 127/a), sx[m] = a/127
 *   GEMM      acc[m,n] = sum_k xq[m,k] W_int8[n,k]   (exact int32)
 *   epilogue  y[m,n] = (fl32(acc) * sw[n]) * sx[m],  sw[n] = smax[n]/127
 *
 * Conventions shared by every entry point:
 *   - Every array pointer is a DEVICE pointer owned by the caller. The library
 *     never allocates, frees or synchronises inside these calls (except
 *     tl_get_status, which synchronises the given stream by design).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and launches on the device current at the call.
 *   - Arrays are row-major and densely packed. Every pointer must be 16-byte
 *     aligned. Argument errors return before anything is launched.
 *   - Shapes: K a positive multiple of 1024 and at most 32768; N a multiple of
 *     128 (N = 0 or M = 0 is a valid empty call that launches nothing).
 *   - Return value: a tl_status code. Errors found on the device (bounded waits
 *     that gave up, codes outside {-1,0,1}) are recorded in a per-device status
 *     word and reported by tl_get_status.
 *   - Weights before activations: the GEMM kernels (tl_linear_prefill,
 *     tl_linear_prefill_noalloc, tl_linear_decode, tl_linear_decode_fused,
 *     tl_linear_decode_f32act) start loading the weight arrays (packed, qT, sw,
 *     s) BEFORE they wait for the preceding kernel in the stream (programmatic
 *     dependent launch), so that the weight stream overlaps that kernel. The
 *     weights must therefore be complete before the preceding kernel in the
 *     stream begins: they must not be written by the kernel launched
 *     immediately before the call. tl_pack_weights meets this by itself (it
 *     ends with a launch that starts only after its outputs are complete), so
 *     its outputs may be used by the very next call; weights written by other
 *     code need any other operation (a kernel, a copy, an event wait) between
 *     the writer and the call. The activations (x, xq, xr, sx) and every output
 *     are touched only after the wait, so they may come from the preceding kernel.
 */
#ifndef TL_H_
#define TL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum tl_status {
  TL_OK = 0,
  TL_EINVAL = 1,        /* NULL pointer, negative size, misaligned pointer, bad dtype */
  TL_EUNSUPPORTED = 2,  /* a shape outside the entry point's range (K % 1024, K > 32768,
                           N % 128, M > 32 on decode; the others' limits are stated with them) */
  TL_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  TL_ETIMEOUT = 4,      /* a bounded device-side wait gave up (via tl_get_status) */
  TL_EDATA = 5,         /* input data out of range, e.g. a code not in {-1,0,1} (via tl_get_status) */
  TL_ENOSPACE = 6       /* a size exceeds the caller-provided capacity */
};

enum tl_dtype {
  TL_I8 = 1,    /* int8 */
  TL_F16 = 2,   /* IEEE binary16 */
  TL_BF16 = 3,  /* bfloat16 */
  TL_F32 = 4    /* IEEE binary32 */
};

/* Human-readable name of a tl_status value (static storage). */
const char* tl_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int tl_version(void);

/*
 * Bytes of the three packed-weight arrays for an N x K layer (Qiita item
 * ecc183fae033565af7cb, 前提: the {-1,0,+1} codes in a 2-bit representation
 * with one fp16 scale per 128 elements; §4 "効いた高速化": the scales as an
 * int8 ratio q per group times a per-row maximum):
 *   packed  N * K / 4  (uint8; 2 bits per code)
 *   qT      (K/128) * N (int8; q transposed, group-major)
 *   sw      N * 4       (fp32; smax / 127 per row)
 * Any output pointer may be NULL. N < 0 or K <= 0 returns TL_EINVAL; K not a
 * multiple of 1024, K > 32768 or N not a multiple of 128 returns TL_EUNSUPPORTED.
 */
int tl_packed_sizes(int N, int K, size_t* packed_bytes, size_t* qT_bytes, size_t* sw_bytes);

/*
 * Load-time weight packing (§4 "効いた高速化": the row-scale decomposition
 * q = round(127 s / smax) and the 2-bit code representation of 前提).
 *
 *   codes   int8 [N, K], values in {-1, 0, +1}
 *   s       fp16 bit patterns [N, K/128]; smax[n] = max_g |s[n,g]|
 *   packed  out: uint32 words [N][K/16] (little endian). Word w of row n
 *           covers k in [16w, 16w+16); the 2-bit field at bit 16h + 2j
 *           holds e = code[n, 16w + 2j + h] + 1 (j = 0..7, h = 0, 1).
 *   qT      out: int8 [K/128, N], qT[g,n] = rne(fl32(fl32(127 s[n,g]) / smax[n]))
 *   sw      out: fp32 [N], sw[n] = fl32(smax[n] / 127); a row with smax = 0
 *           gets q = 0 and sw = 0.
 * A code outside {-1,0,1} records TL_EDATA in the device status word.
 */
int tl_pack_weights(const int8_t* codes, const uint16_t* s, int N, int K,
                    uint8_t* packed, int8_t* qT, float* sw, void* stream);

/*
 * Input-side rotation fused with per-token int8 quantisation (前提: block
 * Hadamard on the input side; §4: per-token int8 after the rotation).
 *
 *   x         bf16 bit patterns [M, K]
 *   signs     optional int8 [K] of +1/-1 applied to x before the rotation
 *             (NULL = all +1)
 *   xq        out [M, K]: the int8 codes; xq_dtype = TL_I8 stores int8 (the
 *             decode path's operand), TL_F16 stores the same integers as
 *             exact fp16 values (the tensor-core operand of tl_linear_prefill
 *             and tl_linear_decode_tc)
 *   sx        out fp32 [M]
 * Per token: xr = fl32 butterflies with strides 1,2,...,512 then x 1/32;
 * a = max |xr|; inv = fl32(127/a); xq = clamp(rne(fl32(xr inv)), +-127);
 * sx = fl32(a/127); a token with a = 0 gives xq = 0 and sx = 0. A token
 * with 0 < a < 127/FLT_MAX (bf16 subnormals only) makes inv = +inf: its
 * non-zero elements code to +-127 and its exact zeros to 0 (the fp32 -> int
 * conversion of the NaN 0 * inf), with sx = fl32(a/127) (possibly 0).
 */
int tl_rotate_quant_act(const uint16_t* x, int M, int K, const int8_t* signs,
                        void* xq, int xq_dtype, float* sx, void* stream);

/*
 * Workspace bytes that let tl_linear_prefill split the K dimension across
 * CTAs (0 when it would not: then every output tile runs whole on one CTA).
 * A problem is split when whole tiles would leave the busiest SM more than
 * six 1024-column chunks above an even share (few tiles with a long K): the
 * tiles of the last partial round of SMs (all of them when there are fewer
 * tiles than SMs) are cut into equal chunk ranges over at most four CTAs per
 * tile, and a cut tile's partial int32 sums meet in a slot of the workspace:
 * one region of 512 bytes per token of the tile for each CTA that may share
 * it (64 KB for a 128-token tile, 8 KB for the 16-token tiles of a batch of
 * at most 16 tokens), plus 32 bytes of counters. With a smaller (or NULL)
 * workspace the call still succeeds, unsplit.
 */
int tl_prefill_workspace_size(int M, int N, int K, size_t* bytes);

/*
 * Prefill (M >= 1) ternary linear layer on the tensor cores (§4: one int8
 * GEMM plus per-row and per-token rescale; the expansion to W_int8 of §6's
 * 31 ms is done inside the GEMM's main loop and never reaches memory).
 *
 *   packed, qT, sw   from tl_pack_weights
 *   xq               fp16 [M, K] holding the int8 codes (tl_rotate_quant_act
 *                    with TL_F16); sx fp32 [M]
 *   y                out [M, N], y_dtype TL_BF16 (rne of the fp32 value) or TL_F32
 *   acc_dbg          optional out int32 [M, N]: the exact integer accumulator
 *   workspace        optional device scratch of ws_bytes (see
 *                    tl_prefill_workspace_size). It must hold zeros before its
 *                    first use (zero it once after allocating it); every call
 *                    that completes leaves it all zero again, so it needs no
 *                    clearing between calls. After a call whose kernel gave up
 *                    (TL_ETIMEOUT from tl_get_status) zero it again. Calls that
 *                    can overlap on the GPU must not share a workspace.
 * Batches of at most 16, 32 or 64 tokens run on tiles of that many tokens (the
 * MMA's N), so that the weights are expanded once for the batch without
 * tensor-core work on padding; larger batches run on 128-token tiles.
 * The integer accumulator is exact: the tensor cores take the int8 values as
 * fp16 (exact), sum each 1024-column block in fp32 (every partial sum is an
 * integer below 127*127*1024 < 2^24, hence exact) and the blocks are added in
 * int32.
 */
int tl_linear_prefill(const uint8_t* packed, const int8_t* qT, const float* sw,
                      const uint16_t* xq, const float* sx, int M, int N, int K,
                      void* y, int y_dtype, int32_t* acc_dbg,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Decode (1 <= M <= 32) ternary linear layer on the CUDA cores (Qiita item
 * ecc183fae033565af7cb §4 "効いた高速化" defines the quantised layer it
 * computes; §5 "効かなかったもの" the int8-activation dp4a decode GEMV it is
 * built on): streams the 2-bit weights once, decodes them in registers and
 * takes int8 dot products (dp4a); same acc and y as tl_linear_prefill, bit
 * for bit.
 *
 *   xq   int8 [M, K] (tl_rotate_quant_act with TL_I8); other arguments as
 *        for tl_linear_prefill. M > 32 returns TL_EUNSUPPORTED.
 * The weights are read before the wait on the preceding kernel (see the
 * conventions above).
 */
int tl_linear_decode(const uint8_t* packed, const int8_t* qT, const float* sw,
                     const int8_t* xq, const float* sx, int M, int N, int K,
                     void* y, int y_dtype, int32_t* acc_dbg, void* stream);

/*
 * Decode (1 <= M <= 32) ternary linear layer on the tensor cores: the same
 * quantised layer (Qiita item ecc183fae033565af7cb §4 "効いた高速化") as
 * tl_linear_decode and tl_linear_prefill, bit for bit, for the decode batch
 * sizes of §5 "効かなかったもの" (the decode GEMV), as mma.sync.m16n8k16 with
 * fp16 operands: each packed word's codes become the fp16 pairs code q exactly
 * (the prefill's expansion, in registers), every 1024-column chunk is summed
 * in fp32 (integers below 2^24, exact) and the chunks in int32.
 *
 *   packed, qT, sw   from tl_pack_weights
 *   xq               fp16 [M, K] holding the int8 codes (tl_rotate_quant_act
 *                    with TL_F16, as for tl_linear_prefill); sx fp32 [M]
 *   y, y_dtype, acc_dbg   as for tl_linear_prefill
 * M > 32 returns TL_EUNSUPPORTED. The weights are read before the wait on the
 * preceding kernel (see the conventions above).
 */
int tl_linear_decode_tc(const uint8_t* packed, const int8_t* qT, const float* sw,
                        const uint16_t* xq, const float* sx, int M, int N, int K, void* y,
                        int y_dtype, int32_t* acc_dbg, void* stream);

/*
 * Decode with the input-side rotation and per-token quantisation done inside
 * the GEMV kernel: equivalent, bit for bit, to tl_rotate_quant_act(x, TL_I8)
 * followed by tl_linear_decode, in one launch (Qiita item
 * ecc183fae033565af7cb: 前提 for the rotation, §4 for the per-token int8 and the
 * row/token rescale, §5 for the dp4a decode GEMV).
 *
 *   x        bf16 bit patterns [M, K]; signs optional int8 [K] (+1/-1)
 *   xq_out   optional int8 [M, K] receiving the quantised tokens (NULL: not written)
 *   sx_out   optional fp32 [M] receiving the token scales (NULL: not written)
 *   other arguments as for tl_linear_decode. M = 0 is a no-op. Supported:
 *   M = 1 with K <= 8192; 2 <= M <= 16 with M' * K <= 73728, M' = M rounded
 *   up to a power of two, and K / 1024 in {1, 2, 3, 4, 5, 8, 16, 17} (the
 *   multi-token decode kernel's shapes: 5 and 8 for M' <= 8, 16 and 17 for
 *   M' <= 4); anything else returns TL_EUNSUPPORTED and launches nothing.
 * The tokens are rotated once per cluster of CTAs, which share them through
 * distributed shared memory; x must be complete when the kernel starts
 * reading it (it waits for the preceding kernel in the stream first).
 */
int tl_linear_decode_fused(const uint8_t* packed, const int8_t* qT, const float* sw,
                           const uint16_t* x, const int8_t* signs, int M, int N, int K, void* y,
                           int y_dtype, int32_t* acc_dbg, int8_t* xq_out, float* sx_out,
                           void* stream);

/*
 * Bytes of the library-owned scratch array used by tl_linear_prefill_noalloc
 * (16 MiB, held on every device that loads the library until the process exits).
 */
#define TL_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * tl_linear_prefill without a caller workspace, for callers that cannot
 * allocate device memory: a host program that has handed all device memory
 * to its own pool (a serving engine that reserves the KV cache up front), or
 * code that must not call cudaMalloc because it synchronises the device.
 * (This entry point has no counterpart on the source pages; it only changes
 * where the scratch lives.)
 *
 * Arguments, layout, result and errors are those of tl_linear_prefill. When
 * the problem has fewer output tiles than SMs, K is split and the partial
 * int32 sums meet in a static device array of TL_NOALLOC_SCRATCH_BYTES owned
 * by the library; the call clears the part it uses before the kernel (so a
 * call that gave up earlier leaves nothing behind for the next). If that
 * part would exceed the array (see tl_prefill_workspace_size) the call returns
 * TL_ENOSPACE and launches nothing, when there are fewer tiles than SMs; with
 * more, a split that does not fit runs every tile whole instead (same
 * result). The call allocates nothing and calls no allocating routine.
 *
 * - Every call shares the one array per device: calls that can overlap on the
 *   GPU (other streams, other host threads) race on it; serialise them.
 * - The first call on a device looks up the array's device address, and the
 *   first prefill call of either entry point on a device loads the library's
 *   kernels together with the array, which reserves its 16 MiB of device memory
 *   and may synchronise the device. Make one call during set-up, before any
 *   stream capture and before the device memory is handed out.
 * - The library caches that address (and its status word's) per device: do not
 *   keep using it after cudaDeviceReset.
 */
int tl_linear_prefill_noalloc(const uint8_t* packed, const int8_t* qT, const float* sw,
                              const uint16_t* xq, const float* sx, int M, int N, int K,
                              void* y, int y_dtype, int32_t* acc_dbg, void* stream);

/*
 * The input-side rotation alone, fp32 out: xr = (1/32) H1024 (signs * x) per
 * 1024-block of each token, the same arithmetic as tl_rotate_quant_act's
 * first step (bit for bit).
 *   x      in  bf16 bit patterns [M, K]; K a multiple of 1024, K <= 32768
 *   signs  in  optional int8 [K] of +1/-1 (NULL: none)
 *   xr     out fp32 [M, K]
 */
int tl_rotate_act(const uint16_t* x, int M, int K, const int8_t* signs, float* xr, void* stream);

/*
 * Decode (1 <= M <= 4) with floating-point activations (Qiita item
 * ecc183fae033565af7cb §5 "効かなかったもの": the production decode kept the
 * activations in floating point and was more exact than the int8 GEMV):
 *   y[m,n] = sum_g s[n,g] sum_{k in g} code[n,k] xr[m,k]
 * in fp32 arithmetic from the packed codes and the ORIGINAL fp16 group scales;
 * no activation quantisation and no int8 q. Same weights as the int8 path
 * (packed from tl_pack_weights) plus s.
 *   packed  in  uint8 [N, K/4] (tl_pack_weights)
 *   s       in  fp16 bit patterns [N, K/128], the scales given to tl_pack_weights
 *   xr      in  fp32 [M, K] (tl_rotate_act)
 *   y       out [M, N], y_dtype TL_F32 or TL_BF16 (rne of the fp32 sum)
 * M > 4 or M * K > 36864 returns TL_EUNSUPPORTED (the activations are staged
 * in shared memory). The sum is in fp32 in an order of the kernel's own; every
 * product code * xr is exact (for |xr| >= 2^-112), so the error is that of
 * at most K/1024 + 23 roundings per term.
 */
int tl_linear_decode_f32act(const uint8_t* packed, const uint16_t* s, const float* xr, int M, int N,
                            int K, void* y, int y_dtype, void* stream);

/*
 * int8 128-group codec of a row-parallel all-reduce payload (Qiita item
 * ecc183fae033565af7cb §6 "最後に残った問題": int8 with one scale per 128
 * elements, all-gathered, each rank adding its own part in bf16; item
 * 66e136acefd5a54b2f1d §5 "解説: 長文を読む速度(prefill)": "compress" and
 * "decompress and add" as one kernel each). The all-gather between the two
 * calls belongs to the caller.
 *
 * tl_codec_quant compresses one part:
 *   x      in  bf16 bit patterns [R, H], row-major; H a multiple of 128
 *   q      out int8 [R, H]
 *   scale  out fp32 [R, H/128]
 * Per 128-element group: a = max |x|; inv = fl32(127/a);
 * q = clamp(rne(fl32(x inv)), -127, 127); scale = fl32(a/127); a = 0 gives
 * q = 0 and scale = 0. A NaN product codes to 0 (what an fp32 -> int
 * conversion gives it); a group whose maximum is below 127/FLT_MAX makes inv
 * +inf, so its non-zero elements code to +-127 and its zeros to 0.
 *
 * tl_codec_dequant_add decompresses the peers' parts and adds them to the own:
 *   own          in  bf16 [R, H], the rank's own part (not compressed)
 *   q_peers      in  int8 [npeers, R, H]; scale_peers fp32 [npeers, R, H/128]
 *   npeers       0..7 (more returns TL_EUNSUPPORTED; 0 copies own to out)
 *   out          out bf16 [R, H]; may be the same buffer as own
 * out = rne_bf16(((own + fl32(q_0 scale_0)) + fl32(q_1 scale_1)) + ...), every
 * product and sum an fp32 operation.
 *
 * Pointers are device pointers, 16-byte aligned; R = 0 is a no-op; H not a
 * multiple of 128 returns TL_EUNSUPPORTED; NULL, misaligned or negative
 * arguments return TL_EINVAL. Nothing is launched on an error.
 */
int tl_codec_quant(const uint16_t* x, int R, int H, int8_t* q, float* scale, void* stream);
int tl_codec_dequant_add(const uint16_t* own, const int8_t* q_peers, const float* scale_peers,
                         int npeers, int R, int H, uint16_t* out, void* stream);

/*
 * Diagnostic: launches one kernel whose bounded wait can never be satisfied (an
 * mbarrier phase nothing arrives at) with a limit of limit_us microseconds
 * (1..100000, else TL_EINVAL). The wait gives up and records TL_ETIMEOUT in
 * the device status word, which the next tl_get_status returns; the CUDA
 * context stays usable. It checks the timeout path every kernel of the
 * library takes when one of its waits runs out (those use a 2 s limit).
 */
int tl_selftest_wait_timeout(unsigned int limit_us, void* stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: TL_OK, TL_ETIMEOUT or TL_EDATA (first error recorded), or TL_ECUDA if
 * the synchronisation itself failed.
 */
int tl_get_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TL_H_ */
