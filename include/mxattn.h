/*
 * mxattn.h -- C ABI of the GB300 (sm_103a) MXAttention forward.
 *
 * The operation is the forward pass of "MXAttention: Data-Free Optimal Scaling
 * and Pre-Normalization Quantization for MXFP4 Attention" (arXiv 2607.24377),
 * Algorithm 2 (section 4.3): a fixed Hadamard rotation of Q and K, MXFP4
 * quantization of Q, K and V with the Universal Optimal Scaling boundary
 * e = ceil(log2(M / 7.25)) (Algorithm 1, Eq. 13/19), and a tiled online
 * softmax (Eqs. 2-8) with Pre-Normalization Quantization of each unnormalized
 * exponential tile (Eqs. 44-48). The causal mode follows the constraint of the
 * MatX note "leaky quantization" (no future token may reach row i).
 *
 * Conventions for every entry point
 *  - Tensors are row-major contiguous [B, H, N, D]; D must be 128.
 *  - Pointers named *_host are host memory; every other pointer is device
 *    memory of the current CUDA device. All device buffers are allocated,
 *    owned and freed by the caller; the library never allocates memory.
 *  - Device pointers must be 16-byte aligned. Inputs must be finite.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Device work
 *    is enqueued asynchronously on it; only mxattn_check and
 *    mxattn_attention_host synchronize.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns a status and enqueues nothing. A launch failure
 *    returns MXATTN_ERR_CUDA. mxattn_last_error() describes the most recent
 *    failure on the calling thread. No C++ exception crosses this boundary.
 *  - B, H or N equal to 0 is an empty problem: MXATTN_OK, nothing launched.
 *  - B*H must not exceed 65535.
 *
 * Quantized layouts (all bytes):
 *  - Q/K codes   [B*H][N][64]: E2M1 codes, channel 2j in the low nibble of
 *                byte j. Code = sign bit (bit 3) + magnitude index into
 *                {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *  - V codes     [B*H][128][Npad/2], Npad = 32*ceil(N/32): channel-major,
 *                token 2j in the low nibble of byte j (the transposed layout
 *                the P.V tensor-core product reads).
 *  - scales      [B*H][ceil(N/128)][512]: biased E8M0 bytes (e + 127), one
 *                512-byte atom per 128-row tile; row r of the tile and
 *                32-element block k sit at byte (r%32)*16 + (r/32)*4 + k.
 *                Rows are tokens for Q/K (blocks = channel blocks) and
 *                channels for V (blocks = 32-token blocks). Slots past N hold
 *                127. An all-zero block has scale byte 127 and zero codes.
 */
#ifndef MXATTN_H
#define MXATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXATTN_API __attribute__((visibility("default")))
#else
#define MXATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXATTN_OK = 0,
  MXATTN_ERR_INVALID_ARG = 1, /* null / misaligned / overlapping pointer, negative size */
  MXATTN_ERR_UNSUPPORTED = 2, /* D != 128, B*H > 65535, N >= 2^31 */
  MXATTN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  MXATTN_ERR_TIMEOUT = 4      /* a kernel's bounded wait expired (reported by mxattn_check) */
} mxattn_status;

/* Byte sizes of the quantized buffers for a [B, H, N, 128] tensor. */
MXATTN_API size_t mxattn_qk_codes_bytes(int64_t B, int64_t H, int64_t N);  /* B*H*N*64 */
MXATTN_API size_t mxattn_qk_scales_bytes(int64_t B, int64_t H, int64_t N); /* B*H*ceil(N/128)*512 */
MXATTN_API size_t mxattn_v_codes_bytes(int64_t B, int64_t H, int64_t N);   /* B*H*128*Npad/2 */
MXATTN_API size_t mxattn_v_scales_bytes(int64_t B, int64_t H, int64_t N);  /* B*H*ceil(N/128)*512 */

/* Algorithm 2 (section 4.3), rotation and Q/K quantization, with Algorithm 1: rotate every token of x by the
 * fixed Hadamard matrix R_H = H_128/sqrt(128) (Sylvester order, binary32
 * butterflies h = 1..64 then one multiply by the binary32 nearest 2^-3.5) and
 * quantize each 32-channel block with the UOS scale.
 *   x      : bf16 [B, H, N, 128] (device, read only)
 *   codes  : mxattn_qk_codes_bytes(B,H,N) bytes (device, written)
 *   scales : mxattn_qk_scales_bytes(B,H,N) bytes (device, written)
 * codes/scales must not overlap x or each other. Used for Q and for K. */
MXATTN_API mxattn_status mxattn_rotate_quantize_qk(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                        void* scales, void* stream);

/* Algorithm 2 (section 4.3), V quantization: quantize V in blocks of 32 consecutive tokens per
 * channel (blocks counted from token 0; the last block is zero padded) with
 * the UOS scale; codes are written channel-major (see layouts above).
 *   v      : bf16 [B, H, N, 128] (device, read only)
 *   codes  : mxattn_v_codes_bytes(B,H,N) bytes; scales: mxattn_v_scales_bytes(B,H,N) bytes */
MXATTN_API mxattn_status mxattn_quantize_v(const void* v, int64_t B, int64_t H, int64_t N, int64_t D, void* codes,
                                void* scales, void* stream);

/* Q, K and V quantized in one launch ("MXAttention" section 5.6: the rotation
 * and the block quantization act on Q/K tiles locally, so they belong in the
 * Q/K preprocessing stage). Writes exactly what mxattn_rotate_quantize_qk(q),
 * mxattn_rotate_quantize_qk(k) and mxattn_quantize_v(v) write, byte for byte,
 * from one kernel with one CTA per SM, in which two warpgroups take the Q and
 * K tiles and a third the V tiles (128 tokens of one head per tile).
 *   q, k, v                            : bf16 [B, H, N, 128] (device, read only)
 *   q_codes/q_scales, k_codes/k_scales : as for mxattn_rotate_quantize_qk
 *   v_codes/v_scales                   : as for mxattn_quantize_v
 * No output may overlap an input or another output (inputs may alias each
 * other). Errors as for the single-tensor calls. */
MXATTN_API mxattn_status mxattn_quantize_qkv(const void* q, const void* k, const void* v, int64_t B, int64_t H,
                                             int64_t N, int64_t D, void* q_codes, void* q_scales, void* k_codes,
                                             void* k_scales, void* v_codes, void* v_scales, void* stream);

/* Algorithm 2 (section 4.3), the attention loop, on quantized operands: for every query row, key
 * tiles of Bc = 128 in increasing order; S = Q^K^T/sqrt(d) and P^V^ on
 * tcgen05 block-scaled MXFP4 tensor cores; running max m, rescale
 * alpha = exp(m_old - m_new); P~ = exp(S - m_new) quantized per 32-key block
 * with the UOS scale (PNQ) and the same P^ feeding both l += sum P^ and
 * O += P^ V^; O = O / l.
 *   q_codes/q_scales, k_codes/k_scales : from mxattn_rotate_quantize_qk
 *   v_codes/v_scales                   : from mxattn_quantize_v
 *   v_bf16 : the unquantized V (bf16 [B,H,N,128]); required when causal,
 *            may be NULL otherwise
 *   causal : 0 = full attention; 1 = key j visible to query i iff j <= i.
 *            For the 32-token V block that contains i, P^ multiplies the
 *            bf16 V rows, so no token after i can influence row i.
 *   out    : fp32 [B, H, N, 128] (device, written) */
MXATTN_API mxattn_status mxattn_forward(const void* q_codes, const void* q_scales, const void* k_codes, const void* k_scales,
                             const void* v_codes, const void* v_scales, const void* v_bf16, int64_t B, int64_t H,
                             int64_t N, int64_t D, int causal, float* out, void* stream);

/* mxattn_forward with the output O = O / l (the finalize step of
 * "MXAttention" Algorithm 2, Eq. 8) written as bf16 instead of fp32: each
 * element is the fp32 value mxattn_forward writes, rounded to the nearest
 * bf16 (ties to even).
 *   out : bf16 [B, H, N, 128] (device, written, 16-byte aligned)
 * Same other arguments and errors as mxattn_forward (causal 0 or 1). */
MXATTN_API mxattn_status mxattn_forward_out_bf16(const void* q_codes, const void* q_scales, const void* k_codes,
                                                 const void* k_scales, const void* v_codes, const void* v_scales,
                                                 const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D,
                                                 int causal, void* out, void* stream);

/* Diagnostic variant of mxattn_forward that also writes every P^ tile:
 *   phat_codes  [B*H][N][ceil(N/128)*64]: E2M1 codes of tile j at bytes
 *               64j..64j+63 (key 2i of the tile in the low nibble of byte i);
 *               tiles a row never visits (causal) are left untouched
 *   phat_scales [B*H][N][ceil(N/128)*4]: biased E8M0 byte of each 32-key block
 * The codes are the ones that enter both l and O (before the causal
 * diagonal-block split). Same arguments and errors as mxattn_forward. */
MXATTN_API mxattn_status mxattn_forward_dump_phat(const void* q_codes, const void* q_scales, const void* k_codes,
                                       const void* k_scales, const void* v_codes, const void* v_scales,
                                       const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                                       float* out, uint8_t* phat_codes, uint8_t* phat_scales, void* stream);

/* BF16 comparison path (no rotation, no quantization): the same online
 * softmax recurrence (Eqs. 2-8) with bf16 Q, K, V and P on tcgen05 kind::f16
 * tensor cores and fp32 accumulation; l sums the bf16-rounded P.
 *   q       : bf16 [B, H, Nq, 128] (device)
 *   k, v    : bf16 [B, H, Nk, 128] (device)
 *   causal  : 0 = every key visible; 1 = key j visible to query i iff j <= i
 *             (both counted from 0)
 *   out     : fp32 [B, H, Nq, 128] (device, written)
 * Nq = 0 (or B*H = 0) is a no-op; Nk = 0 with Nq > 0 is MXATTN_ERR_INVALID_ARG
 * (a softmax over no keys). The sizes obey the limits of mxattn_forward. */
MXATTN_API mxattn_status mxattn_forward_bf16(const void* q, const void* k, const void* v, int64_t B, int64_t H,
                                             int64_t Nq, int64_t Nk, int64_t D, int causal, float* out, void* stream);

/* Ablation variants ("MXAttention" section 5.4, Table 3): the same kernels
 * with the scale rule, the rotation and the placement of l as switches.
 *   rule      : block scale rule of every quantizer it applies to
 *               MXATTN_RULE_UOS: e = ceil(log2(M / 7.25))   (Eq. 13, Algorithm 1)
 *               MXATTN_RULE_OCP: e = floor(log2 M) - 2      (Eq. 11; maxima in [4, 8), above 6 saturate)
 *               MXATTN_RULE_TFS: e = ceil(log2(M / 6))      (Eq. 14)
 *               MXATTN_RULE_CEIL: e = ceil(log2(M / qmax)), qmax in (4, 8]: the
 *                                 Q_max sweep of section 5.5.1 (7.25 is UOS,
 *                                 6 is TFS); qmax is ignored by the other rules
 *               All-zero blocks take sigma = 1 under every rule; e is
 *               clamped to [-127, 127] as for UOS.
 *   rotate    : 1 = fixed Hadamard rotation as in mxattn_rotate_quantize_qk,
 *               0 = quantize the bf16 values as they are
 *   causal    : (mxattn_forward_ex) 0 and 1 as for mxattn_forward; 2 = causal
 *               with the other reading of the MatX note's fix: the query's own
 *               32-token V block is re-quantized per channel over tokens up to
 *               the query only (tokens after it left out of the block maximum),
 *               with the P~ rule p_rule / p_qmax, instead of using the bf16 V
 *               rows; v_bf16 is required for 1 and 2
 *   placement : MXATTN_PLACE_PNQ    l += sum P^ (Eq. 47; what mxattn_forward does)
 *               MXATTN_PLACE_DIRECT l += sum P~, the unquantized exponentials
 *                                   (Eqs. 16-17); O still accumulates P^ V^
 * Layouts, ownership and errors as for the functions they extend; an
 * out-of-range switch returns MXATTN_ERR_INVALID_ARG. With rule = UOS,
 * rotate = 1 and placement = PNQ they compute exactly what
 * mxattn_rotate_quantize_qk, mxattn_quantize_v and mxattn_forward compute.
 * Q and K must share `rotate` (rotating only one changes S). */
typedef enum { MXATTN_RULE_UOS = 0, MXATTN_RULE_OCP = 1, MXATTN_RULE_TFS = 2, MXATTN_RULE_CEIL = 3 } mxattn_scale_rule;
typedef enum { MXATTN_PLACE_PNQ = 0, MXATTN_PLACE_DIRECT = 1 } mxattn_placement;
MXATTN_API mxattn_status mxattn_quantize_qk_ex(const void* x, int64_t B, int64_t H, int64_t N, int64_t D, int rule,
                                               double qmax, int rotate, void* codes, void* scales, void* stream);
MXATTN_API mxattn_status mxattn_quantize_v_ex(const void* v, int64_t B, int64_t H, int64_t N, int64_t D, int rule,
                                              double qmax, void* codes, void* scales, void* stream);
MXATTN_API mxattn_status mxattn_forward_ex(const void* q_codes, const void* q_scales, const void* k_codes,
                                           const void* k_scales, const void* v_codes, const void* v_scales,
                                           const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                                           int p_rule, double p_qmax, int placement, float* out, void* stream);

/* NVFP4 comparison path ("MXAttention" section 1: E2M1 values in 16-element
 * blocks with an E4M3 block scale and a tensor-level scale; section 5.2: the
 * direct NVFP4 baseline quantizes Q, K, V and P~ for the two products, with no
 * smoothing and no softmax-path scaling). Each quantizer first writes the
 * tensor's max |x| to *amax (device float, 4 bytes), then quantizes with the
 * encode factor e_t = fl32(2688 / amax) (2688 = 6 * 448): per block of 16,
 *   sc = E4M3(fl32(fl32(M / 6) * e_t))   (round to nearest even, saturate at 448)
 *   code = E2M1(fl32(x * fl32(e_t / value(sc))))   (every code 0 when sc == 0)
 * Q and K are not rotated. Codes use the MXFP4 layouts (mxattn_qk_codes_bytes,
 * mxattn_v_codes_bytes; V blocks run along tokens). Scales: E4M3 bytes, two
 * 512-byte atoms per 128-row tile (mxattn_nvfp4_scales_bytes), atom kk holding
 * blocks 4kk .. 4kk+3 of row r at byte (r%32)*16 + (r/32)*4 + (block % 4);
 * rows are tokens for Q/K (blocks over channels) and channels for V (blocks
 * over the tile's tokens). Outputs must not overlap the input or each other.
 * Two launches and a 4-byte memset per call, on `stream`. */
MXATTN_API size_t mxattn_nvfp4_scales_bytes(int64_t B, int64_t H, int64_t N); /* B*H*ceil(N/128)*1024 */
MXATTN_API mxattn_status mxattn_nvfp4_quantize_qk(const void* x, int64_t B, int64_t H, int64_t N, int64_t D,
                                                  void* codes, void* scales, float* amax, void* stream);
MXATTN_API mxattn_status mxattn_nvfp4_quantize_v(const void* v, int64_t B, int64_t H, int64_t N, int64_t D,
                                                 void* codes, void* scales, float* amax, void* stream);
/* The attention loop on NVFP4 operands, as the NVFP4 baseline: S from the
 * tcgen05 kind::mxf4nvf4 (scale_vec::4X, UE4M3) product times
 * 1/(e_tQ e_tK); P~ quantized per 16-key block with the E4M3 scale of its
 * maximum / 6 and no tensor scale; O = (P^ V^ / e_tV) / l.
 *   *_codes, *_scales, *_amax : from mxattn_nvfp4_quantize_qk (Q, K) and
 *                               mxattn_nvfp4_quantize_v (V)
 *   causal    : 0, or 1 with the query's own 16-token V block taken from the
 *               bf16 rows (v_bf16 required). The tensor maximum behind e_t is
 *               a statistic of the whole sequence: rows see future tokens
 *               through it unless the maxima are fixed ahead of time.
 *   placement : MXATTN_PLACE_DIRECT (l from P~, the baseline) or
 *               MXATTN_PLACE_PNQ (l from P^)
 *   out       : fp32 [B, H, N, 128] (device)
 * Errors as for mxattn_forward. */
MXATTN_API mxattn_status mxattn_nvfp4_forward(const void* q_codes, const void* q_scales, const float* q_amax,
                                              const void* k_codes, const void* k_scales, const float* k_amax,
                                              const void* v_codes, const void* v_scales, const float* v_amax,
                                              const void* v_bf16, int64_t B, int64_t H, int64_t N, int64_t D,
                                              int causal, int placement, float* out, void* stream);
/* Diagnostic variant of mxattn_nvfp4_forward that also writes every P^ tile,
 * as mxattn_forward_dump_phat does: phat_codes [B*H][N][ceil(N/128)*64]
 * (E2M1 codes, key 2i of a tile in the low nibble of byte i) and
 * phat_scales [B*H][N][ceil(N/128)*8] (the E4M3 byte of each 16-key block). */
MXATTN_API mxattn_status mxattn_nvfp4_forward_dump_phat(const void* q_codes, const void* q_scales,
                                                        const float* q_amax, const void* k_codes,
                                                        const void* k_scales, const float* k_amax,
                                                        const void* v_codes, const void* v_scales,
                                                        const float* v_amax, const void* v_bf16, int64_t B, int64_t H,
                                                        int64_t N, int64_t D, int causal, int placement, float* out,
                                                        uint8_t* phat_codes, uint8_t* phat_scales, void* stream);

/* Device workspace needed by mxattn_attention_host for [B, H, N, 128]. */
MXATTN_API size_t mxattn_workspace_bytes(int64_t B, int64_t H, int64_t N);

/* The whole forward from host memory: copies q/k/v (bf16 [B,H,N,128], host;
 * page-locked memory gives full copy bandwidth and lets the copies overlap
 * the kernels) into `workspace` (device, >= mxattn_workspace_bytes, 256-byte
 * aligned), runs mxattn_quantize_qkv and mxattn_forward, copies the fp32 result to out_host, and synchronizes
 * `stream` before returning, so out_host is ready on MXATTN_OK.
 * The B*H heads run in chunks (the first and the last of one head, the
 * others of about 52 MB of input each, at most 64): each chunk's copy in, kernels and
 * copy out are ordered by events, with the copies on two internal streams
 * and the kernels alternating between `stream` and a third internal stream
 * (all created on the first call on a device and kept). The copies start
 * after the work already queued on `stream`. Calls on the same device from
 * several host threads run one after the other. */
MXATTN_API mxattn_status mxattn_attention_host(const void* q_host, const void* k_host, const void* v_host, int64_t B, int64_t H,
                                    int64_t N, int64_t D, int causal, float* out_host, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* The whole forward (Q, K rotation + quantization, V quantization, attention)
 * for callers that cannot allocate device memory -- for instance an op behind
 * a framework plugin interface that receives only its input and output
 * buffers, or code running under a device-memory budget owned by another
 * allocator. The paper has no counterpart of this entry point.
 * Same arguments as the device-buffer path: q, k, v bf16 [B, H, N, 128],
 * out fp32 [B, H, N, 128] (device, 16-byte aligned, caller-owned).
 * The quantized intermediates live in one fixed device array of the library
 * (mxattn_attention_noalloc_max_scratch_bytes() = 32 MiB), held by every GPU
 * that uses the library until the process exits; problems needing more
 * return MXATTN_ERR_UNSUPPORTED before anything is launched (B*H*N up to about
 * 160 000 token-heads fits). The entry point itself calls no allocator.
 * q, k, v and out must be device memory of the current device (checked with
 * cudaPointerGetAttributes before anything is launched; else
 * MXATTN_ERR_INVALID_ARG).
 * The first call on each device looks up the array's device address with that
 * device current; make that first call before any stream capture. The address
 * is kept for the life of the device's primary context: do not call this
 * entry point on a device after cudaDeviceReset of that device. All calls
 * share the array and it keeps the last call's contents (nothing in it needs
 * clearing: each call rewrites every byte it reads); calls that overlap on the
 * GPU (different streams without ordering, or several host threads) race on
 * it and must be serialized by the caller. */
MXATTN_API mxattn_status mxattn_attention_noalloc(const void* q, const void* k, const void* v, int64_t B, int64_t H,
                                                  int64_t N, int64_t D, int causal, float* out, void* stream);
MXATTN_API size_t mxattn_attention_noalloc_max_scratch_bytes(void);

/* Tensor-core rate probe (measurement only; not a step of the attention).
 * Launches one CTA per SM on `stream`; each issues `iters` iterations of two
 * back-to-back tcgen05.mma kind::mxf4.block_scale.scale_vec::2X, M128 Nn
 * K64, E2M1 operands from shared memory and UE8M0 scales of 2^0 in TMEM, with
 * no other work, so that the caller's event timing of the launch gives the
 * dense FP4 (MXFP4) MMA rate of the device. The rate is the denominator
 * against which the tensor-core share of the attention forward (the QK^T and
 * P^V^ products of "MXAttention", Algorithm 2) is read; n = 128 is the
 * forward's own MMA shape.
 *   iters      1 .. 2^27 iterations per CTA (else MXATTN_ERR_INVALID_ARG).
 *   n          128 or 256 (else MXATTN_ERR_INVALID_ARG).
 *   d_out      optional device float[128*n], written with CTA 0's
 *              accumulator D[r][j] = 128 * iters * a_r * b_j, where a_r is the
 *              E2M1 value of code (7r+1) mod 16 and b_j of code (11j+5) mod 16
 *              (row-major, caller-owned, 4-byte aligned; NULL to skip).
 *   flops_out  optional host double: the launch's FLOP count,
 *              SMs * iters * 2 * (2*128*n*64).
 * A bounded wait that expires sets the status word read by mxattn_check. */
MXATTN_API mxattn_status mxattn_mxf4_mma_rate(int64_t iters, int n, float* d_out, double* flops_out, void* stream);

/* Synchronize `stream`, then read and clear the device status word that the
 * attention kernels set when a bounded wait expires. Returns MXATTN_OK,
 * MXATTN_ERR_TIMEOUT or MXATTN_ERR_CUDA. */
MXATTN_API mxattn_status mxattn_check(void* stream);

/* Test hook. Bit 0 makes the next attention launches skip one internal
 * arrival so that their bounded waits expire (the kernel records
 * MXATTN_ERR_TIMEOUT and returns). 0 restores normal operation. */
MXATTN_API void mxattn_set_debug_flags(uint32_t flags);

/* Message describing the most recent failure on this thread ("" if none). */
MXATTN_API const char* mxattn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MXATTN_H */
