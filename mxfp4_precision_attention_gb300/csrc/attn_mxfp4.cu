// MXFP4 fused attention forward with Pre-Normalization Quantization
// ("MXAttention", Algorithm 2 in section 4.3; Eqs. 2-8 and 44-48).
//
// Per query row, key tiles of Bc = 128 in increasing order:
//   S_j   = Q^ K^_j^T                 tcgen05.mma kind::mxf4 block_scale -> TMEM
//   m_j   = max(m_{j-1}, rowmax S_j / sqrt(d))
//   P~    = exp(S_j / sqrt(d) - m_j)             (registers only)
//   P^    = Q*(P~) per 32-key block, UOS scale   (codes and scales -> TMEM)
//   O     = diag(alpha) O + P^ [V^ | 1]          tcgen05.mma kind::mxf4 -> TMEM
// V^ is extended with 16 rows of ones, so the same MMA that accumulates P^ V^
// also accumulates l = sum P^ in column 128 of the O tile: the row sum and the
// output use the same quantized tile by construction (Eq. 47-48).
//
// A CTA owns two 128-row query tiles (A and B) of one head and streams the
// head's K^/V^ tiles once for both. Warp roles (12 warps):
//   0     TMA producer (Q^ tiles once; K^, V^ tiles + scale atoms, 4-stage rings)
//   1     QK issuer: S = Q^_g K^_j^T for g = A, B alternately into one S buffer
//   2     PV issuer: O_g += P^_g [V^_j | 1]; also owns TMEM
//   3     idle
//   4-7   softmax of tile A, 8-11 softmax of tile B: one full query row per
//         thread (TMEM lanes 32*(w%4)..+31), so no cross-warp reduction is
//         needed, and the two groups run out of phase with each other.
// TMEM (496 of 512 columns): S 128 | O_A 144 | O_B 144 | scale factors 48 |
// P^_A 16 | P^_B 16. The softmax threads write P^ straight into TMEM
// (tcgen05.st): the codes as the A operand of P^V^ (row r in lane r, eight
// E2M1 values per column), the scales where an M=128 block-scaled MMA reads
// row r's A scales (lane r, column base + r/32). The NVFP4 kernels (two scale
// words per operand row, one per K half) keep one buffer of P^ and V^ scales
// to make room for the two P^ operands.
//
// Causal mode (MatX note "leaky quantization"): keys j > i are masked before
// the maximum, tiles past the diagonal are skipped, and for the 32-token V
// block holding the query, P^ multiplies the bf16 V rows instead of V^: the
// block's codes are zeroed in the P^V^ operand, kept by the thread, added to
// l, and multiplied with the diagonal tile's bf16 V rows in the epilogue by
// one kind::f16 tensor-core product into O (causal mode 2, the re-quantized
// diagonal block, does that product on CUDA cores instead).
//
// Every mbarrier wait is bounded (~1 s); on expiry the kernel records an error
// in the device status word, the waiting warp leaves its loop, and TMEM is
// released before the CTA returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr int kThreads = 384;
constexpr int kKStages = 4;
constexpr int kVStages = 4;
constexpr int kOnesRows = 16;                    // extra B rows of ones -> l in column 128
constexpr int kPvN = kD + kOnesRows;             // 144
constexpr uint32_t kTileBytes = kTile * kD / 2;  // 8192 bytes of packed E2M1
constexpr uint32_t kVTileBytes = kPvN * kD / 2;  // 9216

// shared memory carve-up (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                                 // 2 tiles
constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;            // kKStages tiles
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;     // kVStages tiles (+ ones rows)
constexpr uint32_t kOffP = kOffV + kVStages * kVTileBytes;    // [2 groups][2 buffers]: epilogue staging
constexpr int kNumBars = 40;
// Scale atoms, barriers and TMEM scale columns per operand format: MXFP4 has
// one 512-byte atom per 128-row tile (4 blocks of 32 per row, both K halves in
// one 32-bit TMEM word); NVFP4 has two (8 blocks of 16 per row, one word per
// 64-wide MMA).
template <bool kNv, bool kDiag = false>
struct Lay {
  static constexpr uint32_t kSfTile = kNv ? 2 * kSfAtomBytes : kSfAtomBytes;  // scale bytes per tile
  static constexpr uint32_t kOffQSF = kOffP + 4 * kTileBytes;                  // 2 tiles
  static constexpr uint32_t kOffKSF = kOffQSF + 2 * kSfTile;                   // kKStages tiles
  static constexpr uint32_t kOffVSF = kOffKSF + kKStages * kSfTile;            // kVStages tiles
  static constexpr uint32_t kOffOnesSF = kOffVSF + kVStages * kSfTile;         // constant atom: scale 1
  // causal MXFP4 kernels: the diagonal tile's bf16 V and bf16 P^ for the
  // tensor-core diagonal product (128-byte swizzle wants 1024-byte alignment)
  static constexpr uint32_t kOffDiag = (kOffOnesSF + kSfAtomBytes + 1023) / 1024 * 1024;
  static constexpr uint32_t kDiagBytes = kDiag ? 65536 : 0;
  static constexpr uint32_t kOffBars = kDiag ? kOffDiag + kDiagBytes : kOffOnesSF + kSfAtomBytes;
  static constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  // TMEM scale columns (S at 0, O_A and O_B at 128 .. 415)
  //   MXFP4: Q [2 groups] x 4 | K [2 buffers] x 4 | P [2 groups][2 buffers] x 4 | V [2 buffers] x 8
  //   NVFP4, two MMAs (K halves) each: Q [2 groups] x 8 | K [2 buffers] x 8 | P [2 groups] x 8 | V x 16
  //   (its P^ and V^ scales have one buffer: 416 | 432 | 448 | 464)
  static constexpr uint32_t kColSFQ = 416;
  static constexpr uint32_t kColSFK = kNv ? 432 : 424;
  static constexpr uint32_t kColSFP = kNv ? 448 : 432;
  static constexpr uint32_t kColSFV = kNv ? 464 : 448;  // per buffer (x MMA): data atom, then the ones atom at +4
  // the P^ codes of group g (the A operand of its P^V^, 128 keys = 16 columns
  // of eight E2M1 values per row) at kColPT + 16 g
  static constexpr uint32_t kColPT = kNv ? 480 : 464;
  static_assert(kColSFV + 16 <= kColPT && kColPT + 32 <= 512, "TMEM columns overlap");
};

// mbarrier indices
constexpr int kBarQFull = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarVFull = kBarKEmpty + kKStages;
constexpr int kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarSFull = kBarVEmpty + kVStages;  // [2 groups]: S holds S_g of the next tile
constexpr int kBarSEmpty = kBarSFull + 2;         // 4 arrivals: the S buffer was read
constexpr int kBarPFull = kBarSEmpty + 1;         // [2 groups], 4 arrivals: P^ tile + O rescale ready
constexpr int kBarODone = kBarPFull + 2;          // [2 groups]: P^V^ into O_g complete
constexpr int kBarDiagV = kBarODone + 2;          // [2 groups] causal: the group's diagonal bf16 V tile landed
constexpr int kBarDiagP = kBarDiagV + 2;          // [2 groups], 4 arrivals: the group's bf16 P^ rows written
constexpr int kBarDiagDone = kBarDiagP + 2;       // [2 groups]: the diagonal product into O_g complete
static_assert(kBarDiagDone + 2 <= kNumBars, "barrier space");
static_assert(kOffP % 1024 == 0 && kTileBytes % 2048 == 0,
              "the epilogue's staging rows (2 KB per warp and half) are whole 128-byte-swizzle atoms");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kKStages * kTileBytes >= 32768 &&
                  kVStages * kVTileBytes >= 32768,
              "the rings hold group B's diagonal operands (128-byte swizzle, 32 KB each)");

// TMEM columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;                 // O_g at kColO + g * kPvN (144 each)
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2Qmax = 2.8579809951275723f;  // log2(7.25)
constexpr float kLog2Six = 2.5849625007211563f;   // log2(6): TFS scale
constexpr float kExpMagic = 12583039.0f;          // 1.5 * 2^23 + 127

struct Params {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const __nv_bfloat16* v_bf16;
  float* out;
  __nv_bfloat16* out_bf16;  // non-null: O / l is written here as bf16 instead of to `out`
  uint8_t* phat_codes;
  uint8_t* phat_scales;
  int* status;
  int64_t N;
  int NT;
  int causal;
  uint32_t debug_flags;
  int p_rule;     // variant kernels only
  int placement;  // variant kernels only
  float p_log2q;  // variant kernels, kRuleCeilQ: log2(Q_max)
  uint32_t diag_mant_thr;   // causal mode 2: scale rule of the re-quantized diagonal V block
  uint32_t diag_pow2_down;
  float score_scale_log2;  // log2(e) / sqrt(d)
  const float* q_amax;     // NVFP4 kernels: the operands' tensor maxima (device)
  const float* k_amax;
  const float* v_amax;
  int bh_major;  // grid x walks heads and y walks query-tile pairs (causal), else the reverse
};

// two fp32 values -> bf16x2 (round to nearest even), `lo` in the low half
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max over 32 values as a shallow tree of 3-input maxima
__device__ __forceinline__ float max32(const float* v) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; i++) a[i] = fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]), b2 = fmax3(a[6], a[7], a[8]);
  return fmaxf(fmax3(b0, b1, b2), fmaxf(a[9], a[10]));
}

__device__ __forceinline__ float max16(const float* v) {
  const float a0 = fmax3(v[0], v[1], v[2]), a1 = fmax3(v[3], v[4], v[5]), a2 = fmax3(v[6], v[7], v[8]);
  const float a3 = fmax3(v[9], v[10], v[11]), a4 = fmax3(v[12], v[13], v[14]);
  return fmax3(fmax3(a0, a1, a2), fmax3(a3, a4, v[15]), v[15]);
}

constexpr float kSixth = 1.0f / 6.0f;  // binary32 nearest 1/6

// E4M3 codes of two values >= 0 (round to nearest even, saturating at 448):
// lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}
// Values of two E4M3 codes (low byte -> .x), exact through f16.
__device__ __forceinline__ float2 e4m3x2_values(uint32_t h) {
  uint32_t hv;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hv) : "h"(static_cast<uint16_t>(h)));
  return __half22float2(*reinterpret_cast<const __half2*>(&hv));
}

// 1 / e_t with e_t = fl32(2688 / amax), the tensor encode factor of an NVFP4 operand
__device__ __forceinline__ float nv_decode(const float* amax) {
  const float a = __ldg(amax);
  return a > 0.0f ? __frcp_rn(__fdiv_rn(2688.0f, a)) : 1.0f;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float e2m1_decode(uint32_t nib) {
  const uint32_t m = nib & 7u;
  const float mag = (m < 2u) ? 0.5f * static_cast<float>(m)
                             : (1.0f + 0.5f * static_cast<float>(m & 1u)) * static_cast<float>(1u << ((m >> 1) - 1));
  return (nib & 8u) ? -mag : mag;
}

// Four non-negative E2M1 codes (the nibbles of the low 16 bits of c) as two
// bf16x2 words, elements (0, 1) and (2, 3). A non-negative code is a byte
// index 0-7, so one byte permute looks up the high bytes of all four bf16
// values {0, 0.5, 1, 1.5, 2, 3, 4, 6} and one the low bytes.
__device__ __forceinline__ void e2m1x4_bf16(uint32_t c, uint32_t& w01, uint32_t& w23) {
  const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, c);
  const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, c);
  w01 = __byte_perm(lo, hi, 0x5140u);
  w23 = __byte_perm(lo, hi, 0x7362u);
}
// The eight non-negative E2M1 codes of w (element k in nibble k) as binary32.
__device__ __forceinline__ void e2m1x8_f32(uint32_t w, float (&x)[8]) {
  uint32_t b[4];
  e2m1x4_bf16(w & 0xFFFFu, b[0], b[1]);
  e2m1x4_bf16(w >> 16, b[2], b[3]);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    x[2 * i] = __uint_as_float(b[i] << 16);
    x[2 * i + 1] = __uint_as_float(b[i] & 0xFFFF0000u);
  }
}

// Block exponent of a finite maximum M > 0 under a scale rule given by its
// mantissa threshold (the quantizers' rule); denormal maxima clamp to -127.
__device__ __forceinline__ int rule_exponent(float M, uint32_t mant_thr, uint32_t pow2_down) {
  const uint32_t bits = __float_as_uint(M);
  const int b = static_cast<int>(bits >> 23);
  if (b == 0) return -127;
  const uint32_t mant = bits & 0x7FFFFFu;
  const int e = b - 126 - (mant <= mant_thr ? 3 : 2) - ((pow2_down && mant == 0u) ? 1 : 0);
  return e < -127 ? -127 : e;
}

// 2^e as binary32 for e in [-127, 127] (2^-127 is a denormal)
__device__ __forceinline__ float pow2i(int e) {
  return e > -127 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// E2M1 round trip of two values (RNE, saturating at 6): the values the codes stand for
__device__ __forceinline__ float2 e2m1_round2(float y0, float y1) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h)
      : "f"(y0), "f"(y1));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

// kCausal and kDump are compile-time so the non-causal, non-diagnostic path
// carries no checks for either. kVariant builds the ablation variants of
// section 5.4 (Table 3): the P~ blocks take the scale rule p.p_rule (UOS, OCP
// floor of Eq. 11, TFS of Eq. 14, or the ceil rule with a swept Q_max of
// section 5.5.1) and l may come from the unquantized P~
// (direct placement, Eqs. 16-17) instead of P^ (PNQ, Eq. 47).
template <bool kCausal, bool kDump, bool kVariant, bool kNv = false, bool kBf16Out = false>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vb,
                     const __grid_constant__ CUtensorMap tm_o, const Params p) {
  static_assert(!kNv || kVariant, "NVFP4 runs as a variant kernel");
  // causal: the diagonal block's P^ x bf16 V runs on the tensor cores
  constexpr bool kDiagMma = kCausal;
  using L = Lay<kNv, kDiagMma>;
  constexpr uint32_t kOffDiag = L::kOffDiag;
  constexpr uint32_t kOffQSF = L::kOffQSF, kOffKSF = L::kOffKSF, kOffVSF = L::kOffVSF, kOffOnesSF = L::kOffOnesSF;
  constexpr uint32_t kOffBars = L::kOffBars, kOffMisc = L::kOffMisc, kSfTile = L::kSfTile;
  constexpr uint32_t kColSFQ = L::kColSFQ, kColSFK = L::kColSFK, kColSFP = L::kColSFP, kColSFV = L::kColSFV;
  constexpr uint32_t kColPT = L::kColPT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bh = static_cast<int>(p.bh_major ? blockIdx.x : blockIdx.y);
  const int slot = static_cast<int>(p.bh_major ? blockIdx.y : blockIdx.x);
  const int npairs = (p.NT + 1) / 2;
  // causal: heaviest query tiles first
  const int pair = kCausal ? (npairs - 1 - slot) : slot;
  const int qtile0 = 2 * pair, qtile1 = 2 * pair + 1;
  const bool has_b = qtile1 < p.NT;
  const int ntiles0 = kCausal ? qtile0 + 1 : p.NT;
  const int ntiles1 = has_b ? (kCausal ? qtile1 + 1 : p.NT) : 0;
  const int T = ntiles0 > ntiles1 ? ntiles0 : ntiles1;  // key tiles streamed by this CTA
  const int64_t N = p.N;

  // ------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < kKStages; s++) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < kVStages; s++) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int g = 0; g < 2; g++) {
      mbar_init(bar(kBarSFull + g), 1);
      mbar_init(bar(kBarPFull + g), 4);
      mbar_init(bar(kBarODone + g), 1);
    }
    mbar_init(bar(kBarSEmpty), 4);
    if constexpr (kDiagMma) {
      for (int g = 0; g < 2; g++) {
        mbar_init(bar(kBarDiagV + g), 1);
        mbar_init(bar(kBarDiagP + g), 4);
        mbar_init(bar(kBarDiagDone + g), 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_base_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    // constant operand parts: 16 rows of ones (E2M1 1.0 = code 2) under every V
    // stage and the scale atom that goes with them (byte 127 = 2^0)
    const int t = threadIdx.x - 128;
    for (int s = 0; s < kVStages; s++) {
      uint32_t* ones = reinterpret_cast<uint32_t*>(smem + kOffV + s * kVTileBytes + kTileBytes);
      for (int i = t; i < kOnesRows * kD / 8; i += 256) ones[i] = 0x22222222u;
    }
    uint32_t* sf1 = reinterpret_cast<uint32_t*>(smem + kOffOnesSF);
    // scale 1: E8M0 byte 127, or E4M3 byte 0x38
    for (int i = t; i < kSfAtomBytes / 4; i += 256) sf1[i] = kNv ? 0x38383838u : 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  if (warp < 4) {
  if (warp == 0) {
    // --------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      if constexpr (kDiagMma) prefetch_tmap(&tm_vb);
      const int ng = has_b ? 2 : 1;
      mbar_arrive_expect_tx(bar(kBarQFull), ng * (kTileBytes + kSfTile));
      for (int g = 0; g < ng; g++) {
        const int qtg = g ? qtile1 : qtile0;
        tma_load_3d(sb + kOffQ + g * kTileBytes, &tm_q, bar(kBarQFull), 0, qtg * kTile, bh);
        bulk_load(sb + kOffQSF + g * kSfTile, p.q_scales + (static_cast<int64_t>(bh) * p.NT + qtg) * kSfTile, kSfTile,
                  bar(kBarQFull));
      }
      int nk = 0, nv = 0;
      for (int j = 0; j < T; j++) {
        const int ks = j % kKStages, ku = j / kKStages;
        if (ku > 0 && !mbar_wait(bar(kBarKEmpty + ks), (ku - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + ks), kTileBytes + kSfTile);
        tma_load_3d(sb + kOffK + ks * kTileBytes, &tm_k, bar(kBarKFull + ks), 0, j * kTile, bh);
        bulk_load(sb + kOffKSF + ks * kSfTile, p.k_scales + (static_cast<int64_t>(bh) * p.NT + j) * kSfTile, kSfTile,
                  bar(kBarKFull + ks));
        nk++;
        const int vs = j % kVStages, vu = j / kVStages;
        if (vu > 0 && !mbar_wait(bar(kBarVEmpty + vs), (vu - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + vs), kTileBytes + kSfTile);
        tma_load_3d(sb + kOffV + vs * kVTileBytes, &tm_v, bar(kBarVFull + vs), j * (kTile / 2), 0, bh);
        bulk_load(sb + kOffVSF + vs * kSfTile, p.v_scales + (static_cast<int64_t>(bh) * p.NT + j) * kSfTile, kSfTile,
                  bar(kBarVFull + vs));
        nv++;
      }
      // drain: every copy this thread issued must land before the CTA exits
      for (int j = (nk > kKStages ? nk - kKStages : 0); j < nk; j++)
        mbar_wait(bar(kBarKFull + j % kKStages), (j / kKStages) & 1, abort_flag);
      for (int j = (nv > kVStages ? nv - kVStages : 0); j < nv; j++)
        mbar_wait(bar(kBarVFull + j % kVStages), (j / kVStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- QK issuer
    if (lane == 0) {
      const uint32_t id0 = kNv ? idesc_nvf4(128, kTile) : idesc_mxf4(128, kTile, 0, 0);
      const uint32_t id1 = kNv ? idesc_nvf4(128, kTile) : idesc_mxf4(128, kTile, 2, 2);
      // operand descriptors computed once; a stage or buffer moves only the
      // start-address field (16-byte units), which cannot carry out of it here
      const uint64_t dq0 = smem_desc(sb + kOffQ, 16, 512, kSwizzle64B);
      const uint64_t dk0 = smem_desc(sb + kOffK, 16, 512, kSwizzle64B);
      const uint64_t dsfk0 = smem_desc(sb + kOffKSF, 0, 128, kSwizzleNone);
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag);
      if (ok) {
        tc_fence_after();
        if constexpr (kNv) {
          // tile g's atom kk (K half kk) -> columns kColSFQ + 8g + 4kk
          for (int gg = 0; gg < (has_b ? 2 : 1); gg++)
            for (int kk = 0; kk < 2; kk++)
              tc_cp_sf(tmem + kColSFQ + 8 * gg + 4 * kk,
                       smem_desc(sb + kOffQSF + gg * kSfTile + kk * kSfAtomBytes, 0, 128, kSwizzleNone));
        } else {
          tc_cp_sf(tmem + kColSFQ, smem_desc(sb + kOffQSF, 0, 128, kSwizzleNone));
          if (has_b) tc_cp_sf(tmem + kColSFQ + 4, smem_desc(sb + kOffQSF + kSfAtomBytes, 0, 128, kSwizzleNone));
        }
      }
      int n = 0;  // S productions so far
      for (int j = 0; ok && j < T; j++) {
        const int ks = j % kKStages;
        if (!mbar_wait(bar(kBarKFull + ks), (j / kKStages) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sfk = tmem + kColSFK + (kNv ? 8 : 4) * (j & 1);
        tc_cp_sf(sfk, dsfk0 + ks * (kSfTile >> 4));
        if constexpr (kNv) tc_cp_sf(sfk + 4, dsfk0 + ks * (kSfTile >> 4) + (kSfAtomBytes >> 4));
        const uint64_t dk = dk0 + ks * (kTileBytes >> 4);
        for (int g = 0; g < 2; g++) {
          if (j >= (g ? ntiles1 : ntiles0)) continue;
          // the single S buffer is free once the previous production was read
          if (n >= 1 && !mbar_wait(bar(kBarSEmpty), (n - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dq = dq0 + g * (kTileBytes >> 4);
          if constexpr (kNv) {
            const uint32_t sfq = tmem + kColSFQ + 8 * g;
            mma_nvf4(tmem + kColS, dq, dk, id0, sfq, sfk, 0u);
            mma_nvf4(tmem + kColS, dq + 2, dk + 2, id1, sfq + 4, sfk + 4, 1u);  // K step 1: +32 bytes
          } else {
            const uint32_t sfq = tmem + kColSFQ + 4 * g;
            mma_mxf4(tmem + kColS, dq, dk, id0, sfq, sfk, 0u);
            mma_mxf4(tmem + kColS, dq + 2, dk + 2, id1, sfq, sfk, 1u);  // K step 1: +32 bytes
          }
          if (!((p.debug_flags & kDebugNeverArriveS) && n == 0)) tc_commit(bar(kBarSFull + g));
          n++;
        }
        if (!ok) break;
        tc_commit(bar(kBarKEmpty + ks));
      }
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  } else if (warp == 2) {
    // --------------------------------------------------------- PV issuer
    if (lane == 0) {
      const uint32_t id0 = kNv ? idesc_nvf4(128, kPvN) : idesc_mxf4(128, kPvN, 0, 0);
      const uint32_t id1 = kNv ? idesc_nvf4(128, kPvN) : idesc_mxf4(128, kPvN, 2, 2);
      const uint64_t dv0 = smem_desc(sb + kOffV, 16, 512, kSwizzle64B);
      const uint64_t dsfv0 = smem_desc(sb + kOffVSF, 0, 128, kSwizzleNone);
      // scale atom of the ones rows, once into the V scale buffers (each K half for NVFP4)
      if constexpr (kNv) {
        for (int i = 0; i < 2; i++) tc_cp_sf(tmem + kColSFV + 8 * i + 4, smem_desc(sb + kOffOnesSF, 0, 128, kSwizzleNone));
      } else {
        tc_cp_sf(tmem + kColSFV + 4, smem_desc(sb + kOffOnesSF, 0, 128, kSwizzleNone));
        tc_cp_sf(tmem + kColSFV + 12, smem_desc(sb + kOffOnesSF, 0, 128, kSwizzleNone));
      }
      bool ok = true;
      for (int j = 0; ok && j < T; j++) {
        const int vs = j % kVStages;
        if (!mbar_wait(bar(kBarVFull + vs), (j / kVStages) & 1, abort_flag)) { ok = false; break; }
        const uint64_t dv = dv0 + vs * (kVTileBytes >> 4);
        const uint32_t sfv = tmem + kColSFV + (kNv ? 0 : 8 * (j & 1));
        bool sfv_loaded = false;
        for (int g = 0; g < 2; g++) {
          if (j >= (g ? ntiles1 : ntiles0)) continue;
          if (!mbar_wait(bar(kBarPFull + g), j & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          if (!sfv_loaded) {
            // MXFP4: the previous user of this buffer (tile j-2) is complete: the
            // softmax threads waited for it before arriving on p_full. NVFP4 has
            // one buffer, last read by tile j-1's products: its V ring stage's
            // release (committed after them) says they are complete. That
            // barrier's previous phase (tile j-5) completed before the producer
            // refilled the stage for tile j-1, so the parity is unambiguous.
            if (kNv && j >= 1) {
              if (!mbar_wait(bar(kBarVEmpty + (j - 1) % kVStages), ((j - 1) / kVStages) & 1, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            tc_cp_sf(sfv, dsfv0 + vs * (kSfTile >> 4));
            if constexpr (kNv) tc_cp_sf(sfv + 8, dsfv0 + vs * (kSfTile >> 4) + (kSfAtomBytes >> 4));
            sfv_loaded = true;
          }
          const uint32_t od = tmem + kColO + g * kPvN;
          // P^ from TMEM: keys 0-63 in the group's first 8 columns, 64-127 in the next 8
          const uint32_t pa = tmem + kColPT + 16 * g;
          if constexpr (kNv) {
            const uint32_t sfp = tmem + kColSFP + 8 * g;
            mma_nvf4_ta(od, pa, dv, id0, sfp, sfv, j > 0 ? 1u : 0u);
            mma_nvf4_ta(od, pa + 8, dv + 2, id1, sfp + 4, sfv + 8, 1u);
          } else {
            const uint32_t sfp = tmem + kColSFP + 8 * g + 4 * (j & 1);
            mma_mxf4_ta(od, pa, dv, id0, sfp, sfv, j > 0 ? 1u : 0u);
            mma_mxf4_ta(od, pa + 8, dv + 2, id1, sfp, sfv, 1u);
          }
          tc_commit(bar(kBarODone + g));
        }
        if (!ok) break;
        tc_commit(bar(kBarVEmpty + vs));
      }
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  }
  } else {
    // --------------------------------------------------------- softmax
    const int g = (warp - 4) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const int Tg = g ? ntiles1 : ntiles0;
    const int64_t qrow = static_cast<int64_t>(g ? qtile1 : qtile0) * kTile + r;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t ocol = kColO + g * kPvN;
    // NVFP4: S and O carry the tensor encode factors; undo them in C (Q, K) and in the epilogue (V)
    const float C = kNv ? p.score_scale_log2 * nv_decode(p.q_amax) * nv_decode(p.k_amax) : p.score_scale_log2;
    const float vdq = kNv ? nv_decode(p.v_amax) : 1.0f;
    const bool ragged = (N % kTile) != 0;
    float m_run = -INFINITY;
    bool my_abort = false;
    uint32_t diag_words[4] = {0u, 0u, 0u, 0u};  // causal: P^ codes of the query's own 32-key block
    uint32_t diag_sbyte = 127;
    float diag_s = 0.0f;  // NVFP4: E4M3 scale value of the query's own 16-key block
    float l_direct = 0.0f;  // variant kernels, direct placement: l from P~ (Eq. 16)
    bool dv_pending = false;  // causal: this thread's diagonal V load not yet seen to land
    // all lanes poll; the outcome is made warp-uniform so tcgen05 .sync.aligned ops stay convergent
    auto wait_uniform = [&](int b, uint32_t parity) {
      bool ok = !my_abort && mbar_wait(bar(b), parity, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && !my_abort) {
        record_error(p.status, 4, abort_flag);
        my_abort = true;
      }
    };

    for (int j = 0; j < Tg && !my_abort; j++) {
      const int pb = j & 1;
      float v[128];
      uint32_t pw[16];  // the row's P^ codes (eight per word), stored to TMEM after o_done
      uint32_t sfw[2] = {0u, 0u};  // NVFP4: the row's P^ scale words (K halves), stored with the codes
      // the P^ operand of this tile's P^V^ into the group's one TMEM buffer (its
      // last reader, P^V^ of tile j-1, is complete); NVFP4's scale words go with
      // it (one buffer too; MXFP4's are double-buffered and stored earlier).
      // Scales: lane r, column base + r/32 of each K half's word
      auto store_phat = [&]() {
        tmem_st16(tl + kColPT + 16 * g, pw);
        if constexpr (kNv) {
          tmem_st1(tl + kColSFP + 8 * g + quad, sfw[0]);
          tmem_st1(tl + kColSFP + 8 * g + 4 + quad, sfw[1]);
        }
      };
      wait_uniform(kBarSFull + g, j & 1);
      if (my_abort) break;
      tc_fence_after();
      // the row's block maxima (32 keys; NVFP4: 16) from the loads themselves
      float bm_ld[kNv ? 8 : 4];
      if constexpr (kNv) {
        uint32_t r[8][16];
#pragma unroll
        for (int b = 0; b < 8; b++) tmem_ld16_max(tl + kColS + 16 * b, r[b], bm_ld[b]);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 8; b++) {
          uint32_t u = __float_as_uint(bm_ld[b]);
          reg_fence1(u);
          bm_ld[b] = __uint_as_float(u);
#pragma unroll
          for (int i = 0; i < 16; i++) {
            reg_fence1(r[b][i]);
            v[16 * b + i] = __uint_as_float(r[b][i]);
          }
        }
      } else {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32_max(tl + kColS, r0, bm_ld[0]);
        tmem_ld32_max(tl + kColS + 32, r1, bm_ld[1]);
        tmem_ld32_max(tl + kColS + 64, r2, bm_ld[2]);
        tmem_ld32_max(tl + kColS + 96, r3, bm_ld[3]);
        tmem_wait_ld();
        reg_fence32(r0);
        reg_fence32(r1);
        reg_fence32(r2);
        reg_fence32(r3);
#pragma unroll
        for (int b = 0; b < 4; b++) {
          uint32_t u = __float_as_uint(bm_ld[b]);
          reg_fence1(u);
          bm_ld[b] = __uint_as_float(u);
        }
#pragma unroll
        for (int i = 0; i < 32; i++) {
          v[i] = __uint_as_float(r0[i]);
          v[32 + i] = __uint_as_float(r1[i]);
          v[64 + i] = __uint_as_float(r2[i]);
          v[96 + i] = __uint_as_float(r3[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty));

      const bool masked = j == Tg - 1 && (kCausal || ragged);
      uint32_t zmask = 0u;  // MXFP4, non-causal: 0xFF in the byte of each fully masked 32-key block
      if (masked) {
        if constexpr (kDiagMma) {
          // Causal, the group's last (diagonal) key tile: its bf16 V rows for the
          // epilogue's diagonal product start loading now. Group A uses its own
          // 64 KB region. Group B puts them in the K ring: the S just read came
          // from the CTA's last QK^T, so every product that read the ring is
          // complete, and so is every load into it.
          if (!(kVariant && p.causal == 2) && quad == 0 && lane == 0) {
            const uint32_t vdiag = g ? sb + kOffK : sb + kOffDiag;  // [channels 0-63 | 64-127][128 keys][128 B]
            mbar_arrive_expect_tx(bar(kBarDiagV + g), 32768);
            tma_load_3d(vdiag, &tm_vb, bar(kBarDiagV + g), 0, j * kTile, bh);
            tma_load_3d(vdiag + 16384, &tm_vb, bar(kBarDiagV + g), 64, j * kTile, bh);
            dv_pending = true;
          }
        }
        // keys of this tile visible to the row: i < nvalid (key < N, and key <= row if causal)
        const int64_t key0 = static_cast<int64_t>(j) * kTile;
        int64_t lim = N - key0;
        if (kCausal && qrow + 1 - key0 < lim) lim = qrow + 1 - key0;
        const int nvalid = lim < 0 ? 0 : (lim > kTile ? kTile : static_cast<int>(lim));
#pragma unroll
        for (int i = 0; i < 128; i++) v[i] = (i < nvalid) ? v[i] : -INFINITY;
        // the masked keys are -inf in v only: this tile's block maxima come from v
        if constexpr (kNv) {
#pragma unroll
          for (int b = 0; b < 8; b++) bm_ld[b] = max16(v + 16 * b);
        } else {
#pragma unroll
          for (int b = 0; b < 4; b++) {
            bm_ld[b] = max32(v + 32 * b);
            if (!kCausal && bm_ld[b] == -INFINITY) zmask |= 0xFFu << (8 * b);
          }
        }
      }
      float m_new;
      float tile_ptilde = 0.0f;  // direct placement: sum of this row's P~ over the tile
      if constexpr (kNv) {
        // NVFP4 P~ (the comparison baseline): 16-key blocks, E4M3 scale of
        // M/6 where M = 2^((bm - m_new) C) is the block's P~ maximum (exactly 1
        // in the block of the row maximum), no further softmax-path scaling.
        // The offset -log2(S) - m_new C goes into every element's 2^x, so y is
        // P~ / S and its E2M1 code is the block's code.
        float bm[8];
#pragma unroll
        for (int b = 0; b < 8; b++) bm[b] = bm_ld[b];
        m_new = fmax3(fmax3(m_run, bm[0], bm[1]), fmax3(bm[2], bm[3], bm[4]), fmax3(bm[5], bm[6], bm[7]));
        const float mc = m_new * C;
        const bool diag_tile = kCausal && j == Tg - 1;
        const float2 c2 = make_float2(C, C);
        uint8_t* dump = (kDump && qrow < N)
                            ? p.phat_codes + ((static_cast<int64_t>(bh) * N + qrow) * p.NT + j) * 64
                            : nullptr;
        // A block whose scale rounds to 0 (P~ max / 6 below 2^-10) has P^ = 0
        // whatever its codes (the tensor core multiplies them by the zero
        // scale): its y is P~ itself (divisor 1), so that l under direct
        // placement still sums every P~.
        uint32_t sw[2] = {0u, 0u};  // scale bytes of blocks 0-3 (first K half) and 4-7
        float sv[8], sdiv[8], noff[8];
#pragma unroll
        for (int b = 0; b < 8; b += 2) {
          const float2 xm = __fmul2_rn(__fadd2_rn(make_float2(bm[b], bm[b + 1]), make_float2(-m_new, -m_new)), c2);
          const float2 v6 = __fmul2_rn(make_float2(ex2_approx(xm.x), ex2_approx(xm.y)), make_float2(kSixth, kSixth));
          const uint32_t h = e4m3x2(v6.x, v6.y);  // block b in the low byte
          const float2 S = e4m3x2_values(h);
          sv[b] = S.x;
          sv[b + 1] = S.y;
          sdiv[b] = S.x > 0.0f ? S.x : 1.0f;
          sdiv[b + 1] = S.y > 0.0f ? S.y : 1.0f;
          noff[b] = -lg2_approx(sdiv[b]) - mc;
          noff[b + 1] = -lg2_approx(sdiv[b + 1]) - mc;
          sw[b / 4] |= h << (8 * (b % 4));
        }
#pragma unroll
        for (int c = 0; c < 4; c++) {  // 32-key chunk c: blocks 2c and 2c+1
          uint32_t w[4];
#pragma unroll
          for (int hb = 0; hb < 2; hb++) {
            const int b = 2 * c + hb;
            const float2 noff2 = make_float2(noff[b], noff[b]);
            float2 ysum = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int gq = 0; gq < 2; gq++) {
              float y[8];
#pragma unroll
              for (int i = 0; i < 8; i += 2) {
                const float2 x = __ffma2_rn(make_float2(v[16 * b + 8 * gq + i], v[16 * b + 8 * gq + i + 1]), c2, noff2);
                y[i] = ex2_approx(x.x);
                y[i + 1] = ex2_approx(x.y);
                ysum = __fadd2_rn(ysum, make_float2(y[i], y[i + 1]));
              }
              w[2 * hb + gq] = pack_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
            }
            tile_ptilde = fmaf(ysum.x + ysum.y, sdiv[b], tile_ptilde);
          }
          if (kDump && dump != nullptr) *reinterpret_cast<uint4*>(dump + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
          if (diag_tile && c == quad) {
            // the query's own 16-key block (first or second half of the warp's
            // 32 keys): its codes feed the bf16-V product, not the tensor core
            const bool hi = lane >= 16;
            diag_words[0] = hi ? 0u : w[0];
            diag_words[1] = hi ? 0u : w[1];
            diag_words[2] = hi ? w[2] : 0u;
            diag_words[3] = hi ? w[3] : 0u;
            w[0] = hi ? w[0] : 0u;
            w[1] = hi ? w[1] : 0u;
            w[2] = hi ? 0u : w[2];
            w[3] = hi ? 0u : w[3];
            diag_s = hi ? sv[2 * c + 1] : sv[2 * c];
          }
#pragma unroll
          for (int k = 0; k < 4; k++) pw[4 * c + k] = w[k];
        }
        if (kDump && dump != nullptr)
          *reinterpret_cast<uint2*>(p.phat_scales + ((static_cast<int64_t>(bh) * N + qrow) * p.NT + j) * 8) =
              make_uint2(sw[0], sw[1]);
        sfw[0] = sw[0];
        sfw[1] = sw[1];
      } else {
        float bm[4];
#pragma unroll
        for (int b = 0; b < 4; b++) bm[b] = bm_ld[b];
        m_new = fmaxf(fmax3(m_run, bm[0], bm[1]), fmaxf(bm[2], bm[3]));
        const float mc = m_new * C;

        // The TMEM scale columns of parity pb were last read by P^V^ of tile j-2;
        // this thread saw that product complete in its o_done wait of tile j-1.
        // The codes stay in registers until P^V^ of tile j-1, the last reader of
        // the group's one P^ buffer in TMEM, is complete.
        // P^ = Q*(exp(S/sqrt(d) - m_new)) per 32-key block with the UOS scale of the
        // block maximum. Branch-free: a fully masked block has max -inf, all its
        // exponentials are 0 and it takes the all-zero-block scale (byte 127).
        const bool diag_tile = kCausal && j == Tg - 1;
        uint8_t* dump = (kDump && qrow < N)
                            ? p.phat_codes + ((static_cast<int64_t>(bh) * N + qrow) * p.NT + j) * 64
                            : nullptr;
        const float2 c2 = make_float2(C, C);
        // UOS exponents of the four blocks, two at a time on the FMA pipe:
        // e = ceil(max((bm - m_new)*C - log2 7.25, -127)). The block's offset
        // bm - m_new is formed first, so the block holding the row maximum has
        // log2 of its P~ maximum exactly 0 (this matters where a rule's
        // boundary lies on an integer, as for the OCP floor). Adding kExpMagic
        // (1.5*2^23 + 127) rounding toward +inf lands on kExpMagic + e exactly
        // (unit spacing there), so the low byte of its bits is the E8M0 byte
        // e + 127, and kExpMagic - t recovers -e exactly.
        float qoff = kLog2Qmax;
        if constexpr (kVariant)
          qoff = p.p_rule == kRuleTFS ? kLog2Six
                 : p.p_rule == kRuleOCP ? 2.0f
                 : p.p_rule == kRuleCeilQ ? p.p_log2q
                                           : kLog2Qmax;
        const float2 nm2 = make_float2(-m_new, -m_new), nq2 = make_float2(-qoff, -qoff);
        const float2 xe01 = __ffma2_rn(__fadd2_rn(make_float2(bm[0], bm[1]), nm2), c2, nq2);
        const float2 xe23 = __ffma2_rn(__fadd2_rn(make_float2(bm[2], bm[3]), nm2), c2, nq2);
        const float2 mg = make_float2(kExpMagic, kExpMagic);
        float2 t01, t23;
        if (kVariant && p.p_rule == kRuleOCP) {
          // OCP: e = floor(log2 M) - 2, the same add rounding toward -inf
          t01 = __fadd2_rd(make_float2(fmaxf(xe01.x, -127.0f), fmaxf(xe01.y, -127.0f)), mg);
          t23 = __fadd2_rd(make_float2(fmaxf(xe23.x, -127.0f), fmaxf(xe23.y, -127.0f)), mg);
        } else {
          t01 = __fadd2_ru(make_float2(fmaxf(xe01.x, -127.0f), fmaxf(xe01.y, -127.0f)), mg);
          t23 = __fadd2_ru(make_float2(fmaxf(xe23.x, -127.0f), fmaxf(xe23.y, -127.0f)), mg);
        }
        // -(mc + e), rounded once as mc + e would be
        const float2 nmc = make_float2(-mc, -mc), neg1 = make_float2(-1.0f, -1.0f);
        const float2 no01 = __fadd2_rn(__ffma2_rn(t01, neg1, mg), nmc);
        const float2 no23 = __fadd2_rn(__ffma2_rn(t23, neg1, mg), nmc);
        uint32_t sbytes = __byte_perm(__byte_perm(__float_as_uint(t01.x), __float_as_uint(t01.y), 0x0040),
                                      __byte_perm(__float_as_uint(t23.x), __float_as_uint(t23.y), 0x0040), 0x5410);
        // all-zero (fully masked) blocks take sigma = 1. Without causality the
        // blocks were marked where the last tile was masked (a branch here was
        // executed as predicated code in every tile); the causal kernels keep
        // the branch, which times faster there.
        if constexpr (kCausal) {
          if (masked) {
#pragma unroll
            for (int b = 0; b < 4; b++)
              if (bm[b] == -INFINITY) sbytes = (sbytes & ~(0xFFu << (8 * b))) | (127u << (8 * b));
          }
        } else {
          sbytes = (sbytes & ~zmask) | (0x7F7F7F7Fu & zmask);
        }
        // the code loop, compiled twice in the causal kernels: the diagonal tile's
        // copy keeps the query's own block aside, the other tiles' copy carries
        // no trace of it
        auto code_loop = [&](auto diag_c) {
          constexpr bool kDiagTile = decltype(diag_c)::value;
#pragma unroll
        for (int b = 0; b < 4; b++) {
          const float noff = b == 0 ? no01.x : (b == 1 ? no01.y : (b == 2 ? no23.x : no23.y));
          const float2 noff2 = make_float2(noff, noff);
          uint32_t w[4];
          float2 ysum = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int gq = 0; gq < 4; gq++) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              const float2 x = __ffma2_rn(make_float2(v[32 * b + 8 * gq + i], v[32 * b + 8 * gq + i + 1]), c2, noff2);
              y[i] = ex2_approx(x.x);
              y[i + 1] = ex2_approx(x.y);
              if constexpr (kVariant) ysum = __fadd2_rn(ysum, make_float2(y[i], y[i + 1]));
            }
            w[gq] = pack_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
          }
          if constexpr (kVariant) {
            // y = P~ / 2^e of the block; 2^e from the scale byte (byte 0 is 2^-127)
            const uint32_t sb_b = (sbytes >> (8 * b)) & 0xFFu;
            const float scale = sb_b ? __uint_as_float(sb_b << 23) : __uint_as_float(0x00400000u);
            tile_ptilde = fmaf(ysum.x + ysum.y, scale, tile_ptilde);
          }
          if (kDump && dump != nullptr) *reinterpret_cast<uint4*>(dump + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
          if (kDiagTile && b == quad) {
            // the query's own 32-key block: keep its codes for the bf16-V product,
            // drop it from the tensor-core operand
#pragma unroll
            for (int gq = 0; gq < 4; gq++) {
              diag_words[gq] = w[gq];
              w[gq] = 0u;
            }
            diag_sbyte = (sbytes >> (8 * b)) & 0xFFu;
          }
#pragma unroll
          for (int gq = 0; gq < 4; gq++) pw[4 * b + gq] = w[gq];
        }
        };
        if (kCausal && diag_tile)
          code_loop(std::true_type{});
        else
          code_loop(std::false_type{});
        if (kDump && dump != nullptr)
          *reinterpret_cast<uint32_t*>(p.phat_scales + ((static_cast<int64_t>(bh) * N + qrow) * p.NT + j) * 4) = sbytes;
        // P^ scales: lane r, column base + r/32 of this group's scale buffer
        // (the store is waited for with the codes' and O rescale's, before p_full)
        tmem_st1(tl + kColSFP + 8 * g + 4 * pb + quad, sbytes);
      }
      if constexpr (kVariant) l_direct = fmaf(ex2_approx((m_run - m_new) * C), l_direct, tile_ptilde);
      if (j >= 1) {
        // O_g is stable once P^V^ of tile j-1 completes; rescale by alpha if any row's max moved
        const float alpha = ex2_approx((m_run - m_new) * C);
        wait_uniform(kBarODone + g, (j - 1) & 1);
        if (my_abort) break;
        tc_fence_after();
        store_phat();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          // O_g row (128 columns + l) *= alpha: all loads in flight at once, one wait
          const float2 a2 = make_float2(alpha, alpha);
          uint32_t o0[32], o1[32], o2[32], o3[32];
          tmem_ld32(tl + ocol, o0);
          tmem_ld32(tl + ocol + 32, o1);
          tmem_ld32(tl + ocol + 64, o2);
          tmem_ld32(tl + ocol + 96, o3);
          uint32_t l = tmem_ld1(tl + ocol + kD);
          tmem_wait_ld();
          reg_fence32(o0);
          reg_fence32(o1);
          reg_fence32(o2);
          reg_fence32(o3);
          reg_fence1(l);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float2 x;
            x = __fmul2_rn(make_float2(__uint_as_float(o0[i]), __uint_as_float(o0[i + 1])), a2);
            o0[i] = __float_as_uint(x.x);
            o0[i + 1] = __float_as_uint(x.y);
            x = __fmul2_rn(make_float2(__uint_as_float(o1[i]), __uint_as_float(o1[i + 1])), a2);
            o1[i] = __float_as_uint(x.x);
            o1[i + 1] = __float_as_uint(x.y);
            x = __fmul2_rn(make_float2(__uint_as_float(o2[i]), __uint_as_float(o2[i + 1])), a2);
            o2[i] = __float_as_uint(x.x);
            o2[i + 1] = __float_as_uint(x.y);
            x = __fmul2_rn(make_float2(__uint_as_float(o3[i]), __uint_as_float(o3[i + 1])), a2);
            o3[i] = __float_as_uint(x.x);
            o3[i + 1] = __float_as_uint(x.y);
          }
          tmem_st32(tl + ocol, o0);
          tmem_st32(tl + ocol + 32, o1);
          tmem_st32(tl + ocol + 64, o2);
          tmem_st32(tl + ocol + 96, o3);
          tmem_st1(tl + ocol + kD, __float_as_uint(__uint_as_float(l) * alpha));
        }
      } else {
        store_phat();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + g));
      m_run = m_new;
    }

    // --------------------------------------------------------- epilogue
    if (Tg > 0) {
      wait_uniform(kBarODone + g, (Tg - 1) & 1);
      tc_fence_after();
      if (!my_abort) {
        uint32_t lbits = tmem_ld1(tl + ocol + kD);
        tmem_wait_ld();
        reg_fence1(lbits);
        float l = __uint_as_float(lbits);
        // causal: scale of the diagonal block (2^(byte-127), or the E4M3 value)
        const float dsc = kNv ? diag_s : __uint_as_float(diag_sbyte << 23);
        const bool direct = kVariant && p.placement == kPlaceDirect;
        if constexpr (kCausal) {
          // the diagonal block's P^ is not in the tensor-core sum; direct
          // placement already counted its P~
          if (!direct) {
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              float x[8];
              e2m1x8_f32(diag_words[kk], x);
#pragma unroll
              for (int k = 0; k < 8; k++) l += x[k] * dsc;
            }
          }
        }
        if (direct) l = l_direct;
        const float inv_l = 1.0f / l;
        const float inv_lo = kNv ? inv_l * vdq : inv_l;  // O from the tensor cores carries V's encode factor
        // O / l of the warp's 32 rows to global memory in whole 128-byte lines:
        // each 32-column chunk goes through the warp's own rows of the group's
        // two 8 KB staging buffers in shared memory (the region that held P^
        // when it went through shared memory; unused by the key loop), rows
        // 0-15 in the first and 16-31 in the second, 16-byte units swizzled by
        // row % 8 (the 128-byte swizzle of a TMA box). The non-causal kernels
        // then store each half with one TMA copy (rows past N are clipped) and
        // wait for it to read the staging rows before the next chunk; the
        // causal kernels store four rows' 128 bytes per instruction.
        auto store_rows = [&](float inv) {
          uint8_t* stg0 = smem + kOffP + 2 * g * kTileBytes + quad * 2048;
          uint8_t* stg1 = stg0 + kTileBytes;
          const int64_t row0 = qrow - lane;  // global row of the warp's first row
          if constexpr (kBf16Out) {
            // bf16 output: a pass covers 64 columns, again 128 bytes of a row
#pragma unroll 1
            for (int c = 0; c < 2; c++) {
              uint32_t o[32], o2[32];
              tmem_ld32(tl + ocol + 64 * c, o);
              tmem_ld32(tl + ocol + 64 * c + 32, o2);
              tmem_wait_ld();
              reg_fence32(o);
              reg_fence32(o2);
              {
                uint8_t* mine = (lane < 16 ? stg0 : stg1) + (lane & 15) * 128;
                auto pk = [&](const uint32_t* x) {
                  return make_uint4(bf16x2_rn(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                                    bf16x2_rn(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                                    bf16x2_rn(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                                    bf16x2_rn(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
                };
#pragma unroll
                for (int i = 0; i < 4; i++) *reinterpret_cast<uint4*>(mine + ((i ^ (lane & 7)) << 4)) = pk(o + 8 * i);
#pragma unroll
                for (int i = 4; i < 8; i++)
                  *reinterpret_cast<uint4*>(mine + ((i ^ (lane & 7)) << 4)) = pk(o2 + 8 * (i - 4));
              }
              if constexpr (!kCausal) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  if (row0 < N) tma_store_3d(&tm_o, smem_u32(stg0), 128 * c, static_cast<int>(row0), bh);
                  if (row0 + 16 < N) tma_store_3d(&tm_o, smem_u32(stg1), 128 * c, static_cast<int>(row0 + 16), bh);
                  bulk_commit_group();
                  bulk_wait_group_read0();
                }
                __syncwarp();
              } else {
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; it++) {
                  const int i = 4 * it + (lane >> 3), u = lane & 7;
                  const uint4 val = *reinterpret_cast<const uint4*>((i < 16 ? stg0 : stg1) + (i & 15) * 128 + ((u ^ (i & 7)) << 4));
                  if (row0 + i < N)
                    reinterpret_cast<uint4*>(p.out_bf16 + (static_cast<int64_t>(bh) * N + row0 + i) * kD + 64 * c)[u] = val;
                }
                __syncwarp();
              }
            }
          } else {
#pragma unroll 1
            for (int c = 0; c < 4; c++) {
              uint32_t o[32];
              tmem_ld32(tl + ocol + 32 * c, o);
              tmem_wait_ld();
              reg_fence32(o);
              {
                uint8_t* mine = (lane < 16 ? stg0 : stg1) + (lane & 15) * 128;
#pragma unroll
                for (int i = 0; i < 8; i++)
                  *reinterpret_cast<float4*>(mine + ((i ^ (lane & 7)) << 4)) =
                      make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                  __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
              }
              if constexpr (!kCausal) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  if (row0 < N) tma_store_3d(&tm_o, smem_u32(stg0), 128 * c, static_cast<int>(row0), bh);
                  if (row0 + 16 < N) tma_store_3d(&tm_o, smem_u32(stg1), 128 * c, static_cast<int>(row0 + 16), bh);
                  bulk_commit_group();
                  bulk_wait_group_read0();  // the staging rows are rewritten by the next chunk
                }
                __syncwarp();
              } else {
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; it++) {
                  const int i = 4 * it + (lane >> 3), u = lane & 7;
                  const float4 val = *reinterpret_cast<const float4*>((i < 16 ? stg0 : stg1) + (i & 15) * 128 + ((u ^ (i & 7)) << 4));
                  if (row0 + i < N)
                    reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(bh) * N + row0 + i) * kD + 32 * c)[u] = val;
                }
                __syncwarp();  // the staging rows are rewritten by the next chunk
              }
            }
          }
        };
        if constexpr (!kCausal) {
          store_rows(inv_lo);
        } else if (kDiagMma && !(kVariant && p.causal == 2)) {
          // The diagonal block's product on the tensor cores: this row's P^ on its
          // own 32-key block (zero beyond the row and outside the block; exact in
          // bf16, an E2M1 value times a power of two) times the diagonal tile's
          // bf16 V rows (loaded since the group read its last S), one kind::f16
          // 128x128x128 product accumulated into O_g after its last P^V^; every
          // wait is bounded. Group A uses its own 64 KB region. Group B's P^ goes
          // to the V ring: every P^V^ that read it completed before B's last one.
          const uint32_t vdiag = g ? sb + kOffK : sb + kOffDiag;  // [channels 0-63 | 64-127][128 keys][128 B]
          uint8_t* pdiag = g ? smem + kOffV : smem + kOffDiag + 32768;  // [keys 0-63 | 64-127][128 rows][128 B]
          const bool leader = quad == 0 && lane == 0;
          if constexpr (kNv) {
            // O_g holds V^'s encoded units (x e_tV): bring this row to real units
            // first, so the product with the real bf16 V adds in place and the
            // store divides by l only
            const float2 d2 = make_float2(vdq, vdq);
#pragma unroll 1
            for (int c = 0; c < 4; c++) {
              uint32_t o[32];
              tmem_ld32(tl + ocol + 32 * c, o);
              tmem_wait_ld();
              reg_fence32(o);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 y = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), d2);
                o[i] = __float_as_uint(y.x);
                o[i + 1] = __float_as_uint(y.y);
              }
              tmem_st32(tl + ocol + 32 * c, o);
            }
            tmem_wait_st();
          }
          {
            uint32_t pw[16];  // this row's P^ on keys 32*quad .. +31 as bf16 pairs
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              float x[8];
              e2m1x8_f32(diag_words[kk], x);
#pragma unroll
              for (int k = 0; k < 8; k += 2) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[k] * dsc, x[k + 1] * dsc);
                pw[4 * kk + k / 2] = *reinterpret_cast<const uint32_t*>(&h2);
              }
            }
            const int x = r & 7, own_half = quad >> 1, own_c0 = 4 * (quad & 1);
#pragma unroll
            for (int h = 0; h < 2; h++) {
              uint8_t* prow = pdiag + h * 16384 + r * 128;
#pragma unroll
              for (int c = 0; c < 8; c++) {
                const int oc = c - own_c0;
                const bool own = h == own_half && oc >= 0 && oc < 4;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int t = 0; t < 4; t++)
                  if (own && oc == t) val = make_uint4(pw[4 * t], pw[4 * t + 1], pw[4 * t + 2], pw[4 * t + 3]);
                *reinterpret_cast<uint4*>(prow + ((c ^ x) << 4)) = val;
              }
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarDiagP + g));
          if (leader) {
            bool ok = !my_abort && mbar_wait(bar(kBarDiagP + g), 0, abort_flag) &&
                      mbar_wait(bar(kBarDiagV + g), 0, abort_flag);
            dv_pending = dv_pending && !ok;
            if (ok) {
              tc_fence_after();
              const uint32_t idd = idesc_bf16(128, 128, true);
              const uint32_t pa = smem_u32(pdiag);
              for (int i = 0; i < 8; i++)
                mma_bf16(tmem + ocol, smem_desc(pa + (i >> 2) * 16384 + (i & 3) * 32, 16, 1024, kSwizzle128B),
                         smem_desc(vdiag + i * 2048, 16384, 1024, kSwizzle128B), idd, 1u);
            } else {
              record_error(p.status, 4, abort_flag);
            }
            tc_commit(bar(kBarDiagDone + g));  // arrives once the product (if any) is complete
          }
          wait_uniform(kBarDiagDone + g, 0);
          tc_fence_after();
          if (!my_abort) store_rows(inv_l);
        } else {
          // The warp's diagonal block is keys 32*quad .. +31 of tile Tg-1 (its own
          // 32 query rows). Its bf16 V rows pass through shared memory one
          // 32-channel chunk (2 KB) at a time: lane t loads key t's 64 bytes of
          // the chunk, the next chunk's loads are in flight while this one is
          // used, and every thread then reads all 32 rows as broadcasts. The
          // staging space is this group's two 8 KB staging buffers (unused by
          // the key loop): 4 KB per warp, two chunk slots.
          float* orow = p.out + (static_cast<int64_t>(bh) * N + qrow) * kD;
          uint8_t* stage = smem + kOffP + 2 * g * kTileBytes + quad * 4096;
          const int64_t mykey = static_cast<int64_t>(Tg - 1) * kTile + 32 * quad + lane;
          const bool key_ok = mykey < N;
          const uint4* myrow =
              reinterpret_cast<const uint4*>(p.v_bf16) + (static_cast<int64_t>(bh) * N + (key_ok ? mykey : 0)) * (kD / 8);
          const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
          uint4 nxt[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; q4++) nxt[q4] = key_ok ? __ldg(myrow + q4) : zero4;
#pragma unroll 1
          for (int c = 0; c < 4; c++) {
            uint4* slot = reinterpret_cast<uint4*>(stage + (c & 1) * 2048);
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) slot[lane * 4 + q4] = nxt[q4];
            if (c < 3) {
#pragma unroll
              for (int q4 = 0; q4 < 4; q4++) nxt[q4] = key_ok ? __ldg(myrow + 4 * (c + 1) + q4) : zero4;
            }
            // slot c&1 was last read in chunk c-2, before every lane passed the
            // __syncwarp of chunk c-1
            __syncwarp();
            uint32_t o[32];
            tmem_ld32(tl + ocol + 32 * c, o);
            tmem_wait_ld();
            reg_fence32(o);
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; i++) acc[i] = kNv ? __uint_as_float(o[i]) * vdq : __uint_as_float(o[i]);
            if (kVariant && p.causal == 2) {
              // Mode 2: the diagonal V block re-quantized per channel over keys
              // 0..lane (this row's prefix). Lane l reads key l's row; an
              // inclusive prefix-max scan over the lanes gives each row its
              // per-channel block maxima. Keys after the row have P^ = 0.
              float mx[32];
              {
                const uint4* mine = slot + lane * 4;
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                  const uint4 u = mine[q4];
                  const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int t2 = 0; t2 < 4; t2++) {
                    mx[8 * q4 + 2 * t2] = fabsf(__uint_as_float(uu[t2] << 16));
                    mx[8 * q4 + 2 * t2 + 1] = fabsf(__uint_as_float(uu[t2] & 0xFFFF0000u));
                  }
                }
              }
#pragma unroll
              for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int i = 0; i < 32; i++) {
                  const float other = __shfl_up_sync(0xffffffffu, mx[i], d);
                  if (lane >= d) mx[i] = fmaxf(mx[i], other);
                }
              }
              float inv[32], t[32];
#pragma unroll
              for (int i = 0; i < 32; i++) {
                const int e = mx[i] > 0.0f ? rule_exponent(mx[i], p.diag_mant_thr, p.diag_pow2_down) : 0;
                inv[i] = pow2i(-e);
                t[i] = 0.0f;
              }
#pragma unroll 1
              for (int kk = 0; kk < 4; kk++) {
                const uint32_t wk = kk == 0 ? diag_words[0] : (kk == 1 ? diag_words[1] : (kk == 2 ? diag_words[2] : diag_words[3]));
#pragma unroll
                for (int k = 0; k < 8; k++) {
                  const float pk = e2m1_decode((wk >> (4 * k)) & 0xFu) * dsc;
                  const uint4* vr = slot + (8 * kk + k) * 4;
#pragma unroll
                  for (int q4 = 0; q4 < 4; q4++) {
                    const uint4 u = vr[q4];
                    const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int t2 = 0; t2 < 4; t2++) {
                      const int c0 = 8 * q4 + 2 * t2;
                      const float2 y = __fmul2_rn(make_float2(__uint_as_float(uu[t2] << 16), __uint_as_float(uu[t2] & 0xFFFF0000u)),
                                                  make_float2(inv[c0], inv[c0 + 1]));
                      const float2 dq = e2m1_round2(y.x, y.y);
                      const float2 r = __ffma2_rn(make_float2(pk, pk), dq, make_float2(t[c0], t[c0 + 1]));
                      t[c0] = r.x;
                      t[c0 + 1] = r.y;
                    }
                  }
                }
              }
              // 2^e = 1 / 2^-e exactly (IEEE reciprocal of a power of two)
#pragma unroll
              for (int i = 0; i < 32; i++) acc[i] = fmaf(__frcp_rn(inv[i]), t[i], acc[i]);
            } else {
            // masked keys (beyond the row or beyond N) have P^ = 0; their staged
            // rows are finite (zeros past N)
#pragma unroll 1
            for (int kk = 0; kk < 4; kk++) {
              const uint32_t wk = kk == 0 ? diag_words[0] : (kk == 1 ? diag_words[1] : (kk == 2 ? diag_words[2] : diag_words[3]));
#pragma unroll
              for (int k = 0; k < 8; k++) {
                const float pk = e2m1_decode((wk >> (4 * k)) & 0xFu) * dsc;
                const uint4* vr = slot + (8 * kk + k) * 4;
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                  const uint4 u = vr[q4];
                  const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int t2 = 0; t2 < 4; t2++) {
                    acc[8 * q4 + 2 * t2] = fmaf(pk, __uint_as_float(uu[t2] << 16), acc[8 * q4 + 2 * t2]);
                    acc[8 * q4 + 2 * t2 + 1] = fmaf(pk, __uint_as_float(uu[t2] & 0xFFFF0000u), acc[8 * q4 + 2 * t2 + 1]);
                  }
                }
              }
            }
            }
            if (qrow < N) {
              float4* dst = reinterpret_cast<float4*>(orow + 32 * c);
#pragma unroll
              for (int i = 0; i < 8; i++)
                dst[i] = make_float4(acc[4 * i] * inv_l, acc[4 * i + 1] * inv_l, acc[4 * i + 2] * inv_l,
                                     acc[4 * i + 3] * inv_l);
            }
          }
        }
      }
    }
    // after an abort, a diagonal V load issued in the last key tile must land
    // before the CTA exits (bounded, like every wait)
    if (dv_pending) mbar_wait(bar(kBarDiagV + g), 0, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_mxfp4_forward(const Mxfp4FwdArgs& a, cudaStream_t s) {
  const int64_t N = a.N, BH = a.BH;
  const int64_t NT = ceil_div(N, kTile);
  const int64_t npad_bytes = ceil_div(N, kBlock) * kBlock / 2;
  alignas(64) CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {64, static_cast<uint64_t>(N) * 64};
    const uint32_t box[3] = {64, kTile, 1};
    if (!encode_tensor_map(&tq, 0, 3, const_cast<void*>(a.q_codes), dims, strides, box, 64)) return cudaErrorInvalidValue;
    if (!encode_tensor_map(&tk, 0, 3, const_cast<void*>(a.k_codes), dims, strides, box, 64)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(npad_bytes), static_cast<uint64_t>(kD), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(npad_bytes), static_cast<uint64_t>(npad_bytes) * kD};
    const uint32_t box[3] = {64, kD, 1};
    if (!encode_tensor_map(&tv, 0, 3, const_cast<void*>(a.v_codes), dims, strides, box, 64)) return cudaErrorInvalidValue;
  }
  // the bf16 V for the causal diagonal tile (the same map shape as the BF16 path)
  alignas(64) CUtensorMap tvb = tv;
  if (a.causal && a.v_bf16 != nullptr) {
    const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {static_cast<uint64_t>(kD) * 2, static_cast<uint64_t>(N) * kD * 2};
    const uint32_t box[3] = {64, kTile, 1};
    if (!encode_tensor_map(&tvb, 1, 3, const_cast<void*>(a.v_bf16), dims, strides, box, 128))
      return cudaErrorInvalidValue;
  }
  alignas(64) CUtensorMap to;
  {
    const bool ob = a.out_bf16 != nullptr;
    const uint64_t row = ob ? kD * 2 : kD * 4;
    const uint64_t dims[3] = {row, static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {row, static_cast<uint64_t>(N) * row};
    const uint32_t box[3] = {128, 16, 1};
    if (!encode_tensor_map(&to, 0, 3, ob ? a.out_bf16 : static_cast<void*>(a.out), dims, strides, box, 128))
      return cudaErrorInvalidValue;
  }
  Params p;
  p.q_scales = static_cast<const uint8_t*>(a.q_scales);
  p.k_scales = static_cast<const uint8_t*>(a.k_scales);
  p.v_scales = static_cast<const uint8_t*>(a.v_scales);
  p.v_bf16 = static_cast<const __nv_bfloat16*>(a.v_bf16);
  p.out = a.out;
  p.out_bf16 = static_cast<__nv_bfloat16*>(a.out_bf16);
  p.phat_codes = a.phat_codes;
  p.phat_scales = a.phat_scales;
  p.status = device_status_ptr();
  p.N = N;
  p.NT = static_cast<int>(NT);
  p.causal = a.causal;
  p.debug_flags = a.debug_flags;
  p.p_rule = a.p_rule;
  p.placement = a.placement;
  p.p_log2q = static_cast<float>(std::log2(a.p_qmax));
  rule_threshold(a.p_rule, a.p_qmax, &p.diag_mant_thr, &p.diag_pow2_down);
  p.score_scale_log2 = kLog2e / 11.313708498984761f;  // log2(e) / sqrt(128)
  p.q_amax = a.q_amax;
  p.k_amax = a.k_amax;
  p.v_amax = a.v_amax;
  const bool nv = a.q_amax != nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  constexpr uint32_t kSmemMx = Lay<false>::kSmemBytes, kSmemNv = Lay<true>::kSmemBytes;
  constexpr uint32_t kSmemMxC = Lay<false, true>::kSmemBytes;  // causal: + the diagonal tiles
  constexpr uint32_t kSmemNvC = Lay<true, true>::kSmemBytes;
  if (!attr_set[dev]) {
    for (auto fn : {mxfp4_fwd_kernel<false, false, false>, mxfp4_fwd_kernel<false, true, false>,
                    mxfp4_fwd_kernel<false, false, true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMx);
      if (e != cudaSuccess) return e;
    }
    for (auto fn : {mxfp4_fwd_kernel<true, false, false>, mxfp4_fwd_kernel<true, true, false>,
                    mxfp4_fwd_kernel<true, false, true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMxC);
      if (e != cudaSuccess) return e;
    }
    for (auto fn : {mxfp4_fwd_kernel<false, false, true, true>, mxfp4_fwd_kernel<false, true, true, true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemNv);
      if (e != cudaSuccess) return e;
    }
    for (auto fn : {mxfp4_fwd_kernel<true, false, true, true>, mxfp4_fwd_kernel<true, true, true, true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemNvC);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(mxfp4_fwd_kernel<false, false, false, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMx);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mxfp4_fwd_kernel<true, false, false, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMxC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // Blocks start in grid order, x fastest. Non-causal items all cost the same, and
  // putting the pairs of one head side by side keeps that head's K/V hot in L2.
  // Causal items cost 2*pair + 2 key tiles: with heads on x every head's longest
  // pair starts first and the short ones fill the last wave (longest first).
  const int64_t npairs = (NT + 1) / 2;
  p.bh_major = (a.causal && npairs <= 65535) ? 1 : 0;
  dim3 grid = p.bh_major ? dim3(static_cast<unsigned>(BH), static_cast<unsigned>(npairs))
                         : dim3(static_cast<unsigned>(npairs), static_cast<unsigned>(BH));
  const bool dump = a.phat_codes != nullptr;
  const bool variant = a.p_rule != kRuleUOS || a.placement != kPlacePNQ || a.causal == 2;
  if (!nv && variant && dump) return cudaErrorNotSupported;  // the MXFP4 P^ dump covers UOS + PNQ only
  if (nv && (a.causal == 2 || a.p_rule != kRuleUOS)) return cudaErrorNotSupported;
  if (a.out_bf16 != nullptr) {  // bf16 output: the plain MXFP4 kernels only (UOS, PNQ, no dump)
    if (nv || variant || dump) return cudaErrorNotSupported;
    if (a.causal) mxfp4_fwd_kernel<true, false, false, false, true><<<grid, kThreads, kSmemMxC, s>>>(tq, tk, tv, tvb, to, p);
    else mxfp4_fwd_kernel<false, false, false, false, true><<<grid, kThreads, kSmemMx, s>>>(tq, tk, tv, tvb, to, p);
    return cudaGetLastError();
  }
  if (nv) {
    if (a.causal) {
      if (dump) mxfp4_fwd_kernel<true, true, true, true><<<grid, kThreads, kSmemNvC, s>>>(tq, tk, tv, tvb, to, p);
      else mxfp4_fwd_kernel<true, false, true, true><<<grid, kThreads, kSmemNvC, s>>>(tq, tk, tv, tvb, to, p);
    } else {
      if (dump) mxfp4_fwd_kernel<false, true, true, true><<<grid, kThreads, kSmemNv, s>>>(tq, tk, tv, tvb, to, p);
      else mxfp4_fwd_kernel<false, false, true, true><<<grid, kThreads, kSmemNv, s>>>(tq, tk, tv, tvb, to, p);
    }
  } else if (variant) {
    if (a.causal) mxfp4_fwd_kernel<true, false, true><<<grid, kThreads, kSmemMxC, s>>>(tq, tk, tv, tvb, to, p);
    else mxfp4_fwd_kernel<false, false, true><<<grid, kThreads, kSmemMx, s>>>(tq, tk, tv, tvb, to, p);
  } else if (a.causal) {
    if (dump) mxfp4_fwd_kernel<true, true, false><<<grid, kThreads, kSmemMxC, s>>>(tq, tk, tv, tvb, to, p);
    else mxfp4_fwd_kernel<true, false, false><<<grid, kThreads, kSmemMxC, s>>>(tq, tk, tv, tvb, to, p);
  } else {
    if (dump) mxfp4_fwd_kernel<false, true, false><<<grid, kThreads, kSmemMx, s>>>(tq, tk, tv, tvb, to, p);
    else mxfp4_fwd_kernel<false, false, false><<<grid, kThreads, kSmemMx, s>>>(tq, tk, tv, tvb, to, p);
  }
  return cudaGetLastError();
}

}  // namespace mxattn
