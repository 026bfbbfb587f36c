// MXFP4 fused attention forward with Pre-Normalization Quantization
// ("MXAttention", Algorithm 2 lines 8-21; Eqs. 2-8 and 44-48).
//
// One CTA owns one 128-row query tile of one head and walks the key tiles
// (Bc = 128) in increasing order:
//   S_j   = Q^ K^_j^T                 tcgen05.mma kind::mxf4 block_scale -> TMEM
//   m_new = max(m, rowmax S_j / sqrt(d))
//   P~    = exp(S_j / sqrt(d) - m_new)           (registers only)
//   P^    = Q*(P~) per 32-key block, UOS scale   (codes + scales -> smem)
//   O     = diag(alpha) O + P^ [V^ | 1]          tcgen05.mma kind::mxf4 -> TMEM
// V^ is extended with 16 rows of ones, so the same MMA that accumulates P^ V^
// also accumulates l = sum P^ in column 128 of the O tile: the row sum and the
// output use the same quantized tile by construction (Eq. 47-48).
//
// Warp roles (12 warps): 0 = TMA producer, 1 = MMA issuer + TMEM owner,
// 2-3 idle, 4-11 = softmax. Softmax warp w handles TMEM lanes 32*(w%4)..+31
// (one query row per thread) and key half h = (w-4)/4 of every tile (keys
// 64h..64h+63), exchanging row maxima with the other half through smem.
//
// Causal mode (MatX note "leaky quantization"): keys j > i are masked before
// the maximum, tiles past the diagonal are skipped, and for the 32-token V
// block holding the query, P^ multiplies the bf16 V rows instead of V^ (that
// product is formed on CUDA cores in the epilogue; the block's P^ codes are
// zeroed in the tensor-core operand and its sum is added to l separately).
//
// Every mbarrier wait is bounded (~1 s); on expiry the kernel records an error
// in the device status word, votes all softmax threads out of the loop, and
// releases TMEM before returning.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr int kThreads = 384;
constexpr int kKStages = 4;
constexpr int kVStages = 4;
constexpr int kOnesRows = 16;                   // extra B rows of ones -> l in column 128
constexpr int kPvN = kD + kOnesRows;            // 144
constexpr uint32_t kTileBytes = kTile * kD / 2;  // 8192 bytes of packed E2M1
constexpr uint32_t kVTileBytes = kPvN * kD / 2;  // 9216

// shared memory carve-up (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kVStages * kVTileBytes;
constexpr uint32_t kOffQSF = kOffP + 2 * kTileBytes;
constexpr uint32_t kOffKSF = kOffQSF + kSfAtomBytes;
constexpr uint32_t kOffVSF = kOffKSF + kKStages * kSfAtomBytes;
constexpr uint32_t kOffPSF = kOffVSF + kVStages * 2 * kSfAtomBytes;
constexpr uint32_t kOffXchg = kOffPSF + 2 * kSfAtomBytes;   // [2 buf][2 half][128] float
constexpr uint32_t kOffLsum = kOffXchg + 2 * 2 * kTile * 4;
constexpr uint32_t kOffLx = kOffLsum + kTile * 4;
constexpr int kPdiagStride = 33;                             // floats per row (+1 pad)
constexpr uint32_t kOffPdiag = kOffLx + kTile * 4;
constexpr uint32_t kOffVdiag = kOffPdiag + kTile * kPdiagStride * 4;  // bf16 [128][128]
constexpr uint32_t kOffBars = kOffVdiag + kTile * kD * 2;
constexpr int kNumBars = 32;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack

// mbarrier indices
constexpr int kBarQFull = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarVFull = kBarKEmpty + kKStages;
constexpr int kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarSFull = kBarVEmpty + kVStages;
constexpr int kBarSEmpty = kBarSFull + 2;
constexpr int kBarPFull = kBarSEmpty + 2;
constexpr int kBarPEmpty = kBarPFull + 2;
constexpr int kBarODone = kBarPEmpty + 2;
static_assert(kBarODone < kNumBars, "barrier space");

// TMEM columns
constexpr uint32_t kColS = 0;      // 2 x 128
constexpr uint32_t kColO = 256;    // 144
constexpr uint32_t kColSFQ = 400;  // 4
constexpr uint32_t kColSFK = 404;  // 2 x 4
constexpr uint32_t kColSFP = 412;  // 2 x 4
constexpr uint32_t kColSFV = 420;  // 2 x 8
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2Qmax = 2.8579809951275723f;  // log2(7.25)

struct Params {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const __nv_bfloat16* v_bf16;
  float* out;
  uint8_t* phat_codes;
  uint8_t* phat_scales;
  int* status;
  int64_t N;
  int NT;
  int causal;
  uint32_t debug_flags;
  float score_scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float e2m1_decode(uint32_t nib) {
  const uint32_t m = nib & 7u;
  const float mag = (m < 2u) ? 0.5f * static_cast<float>(m)
                             : (1.0f + 0.5f * static_cast<float>(m & 1u)) * static_cast<float>(1u << ((m >> 1) - 1));
  return (nib & 8u) ? -mag : mag;
}

__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bh = blockIdx.y;
  // causal: heaviest query tiles first
  const int qt = p.causal ? (p.NT - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int T = p.causal ? qt + 1 : p.NT;
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
    for (int b = 0; b < 2; b++) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarSEmpty + b), 8);
      mbar_init(bar(kBarPFull + b), 8);
      mbar_init(bar(kBarPEmpty + b), 1);
    }
    mbar_init(bar(kBarODone), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_base_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    // constant parts of every V stage: 16 rows of ones (E2M1 1.0 = code 2) and
    // their scale atom (byte 127 = 2^0); also the P^ diagonal scratch.
    const int t = threadIdx.x - 128;
    for (int s = 0; s < kVStages; s++) {
      uint32_t* ones = reinterpret_cast<uint32_t*>(smem + kOffV + s * kVTileBytes + kTileBytes);
      for (int i = t; i < kOnesRows * kD / 8; i += 256) ones[i] = 0x22222222u;
      uint32_t* sf1 = reinterpret_cast<uint32_t*>(smem + kOffVSF + s * 2 * kSfAtomBytes + kSfAtomBytes);
      for (int i = t; i < kSfAtomBytes / 4; i += 256) sf1[i] = 0x7F7F7F7Fu;
    }
    reinterpret_cast<float*>(smem + kOffLx)[t % kTile] = 0.0f;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;

  if (warp == 0) {
    // --------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQFull), kTileBytes + kSfAtomBytes);
      tma_load_3d(sb + kOffQ, &tm_q, bar(kBarQFull), 0, qt * kTile, bh);
      bulk_load(sb + kOffQSF, p.q_scales + (static_cast<int64_t>(bh) * p.NT + qt) * kSfAtomBytes, kSfAtomBytes,
                bar(kBarQFull));
      int nk = 0, nv = 0;
      for (int j = 0; j < T; j++) {
        const int ks = j % kKStages, ku = j / kKStages;
        if (ku > 0 && !mbar_wait(bar(kBarKEmpty + ks), (ku - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + ks), kTileBytes + kSfAtomBytes);
        tma_load_3d(sb + kOffK + ks * kTileBytes, &tm_k, bar(kBarKFull + ks), 0, j * kTile, bh);
        bulk_load(sb + kOffKSF + ks * kSfAtomBytes,
                  p.k_scales + (static_cast<int64_t>(bh) * p.NT + j) * kSfAtomBytes, kSfAtomBytes,
                  bar(kBarKFull + ks));
        nk++;
        const int vs = j % kVStages, vu = j / kVStages;
        if (vu > 0 && !mbar_wait(bar(kBarVEmpty + vs), (vu - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + vs), kTileBytes + kSfAtomBytes);
        tma_load_3d(sb + kOffV + vs * kVTileBytes, &tm_v, bar(kBarVFull + vs), j * (kTile / 2), 0, bh);
        bulk_load(sb + kOffVSF + vs * 2 * kSfAtomBytes,
                  p.v_scales + (static_cast<int64_t>(bh) * p.NT + j) * kSfAtomBytes, kSfAtomBytes,
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
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s0 = idesc_mxf4(128, kTile, 0, 0), idesc_s1 = idesc_mxf4(128, kTile, 2, 2);
      const uint32_t idesc_o0 = idesc_mxf4(128, kPvN, 0, 0), idesc_o1 = idesc_mxf4(128, kPvN, 2, 2);
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag);
      if (ok) {
        tc_fence_after();
        tc_cp_sf(tmem + kColSFQ, smem_desc(sb + kOffQSF, 0, 128, kSwizzleNone));
      }
      auto issue_pv = [&](int t) -> bool {
        const int pb = t & 1, vs = t % kVStages;
        if (!mbar_wait(bar(kBarPFull + pb), (t >> 1) & 1, abort_flag)) return false;
        if (!mbar_wait(bar(kBarVFull + vs), (t / kVStages) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t sfp = tmem + kColSFP + 4 * pb, sfv = tmem + kColSFV + 8 * pb;
        tc_cp_sf(sfp, smem_desc(sb + kOffPSF + pb * kSfAtomBytes, 0, 128, kSwizzleNone));
        tc_cp_sf(sfv, smem_desc(sb + kOffVSF + vs * 2 * kSfAtomBytes, 0, 128, kSwizzleNone));
        tc_cp_sf(sfv + 4, smem_desc(sb + kOffVSF + vs * 2 * kSfAtomBytes + kSfAtomBytes, 0, 128, kSwizzleNone));
        const uint32_t pa = sb + kOffP + pb * kTileBytes, va = sb + kOffV + vs * kVTileBytes;
        mma_mxf4(tmem + kColO, smem_desc(pa, 16, 512, kSwizzle64B), smem_desc(va, 16, 512, kSwizzle64B), idesc_o0,
                 sfp, sfv, t > 0 ? 1u : 0u);
        mma_mxf4(tmem + kColO, smem_desc(pa + 32, 16, 512, kSwizzle64B), smem_desc(va + 32, 16, 512, kSwizzle64B),
                 idesc_o1, sfp, sfv, 1u);
        tc_commit(bar(kBarODone));
        tc_commit(bar(kBarPEmpty + pb));
        tc_commit(bar(kBarVEmpty + vs));
        return true;
      };
      for (int j = 0; ok && j < T; j++) {
        const int ks = j % kKStages, s = j & 1;
        if (!mbar_wait(bar(kBarKFull + ks), (j / kKStages) & 1, abort_flag)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sfk = tmem + kColSFK + 4 * s;
        tc_cp_sf(sfk, smem_desc(sb + kOffKSF + ks * kSfAtomBytes, 0, 128, kSwizzleNone));
        const uint32_t ka = sb + kOffK + ks * kTileBytes, qa = sb + kOffQ;
        mma_mxf4(tmem + kColS + s * kTile, smem_desc(qa, 16, 512, kSwizzle64B), smem_desc(ka, 16, 512, kSwizzle64B),
                 idesc_s0, tmem + kColSFQ, sfk, 0u);
        mma_mxf4(tmem + kColS + s * kTile, smem_desc(qa + 32, 16, 512, kSwizzle64B),
                 smem_desc(ka + 32, 16, 512, kSwizzle64B), idesc_s1, tmem + kColSFQ, sfk, 1u);
        if (!((p.debug_flags & kDebugNeverArriveS) && j == 0)) tc_commit(bar(kBarSFull + s));
        tc_commit(bar(kBarKEmpty + ks));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !issue_pv(T - 1)) ok = false;
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  } else if (warp >= 4) {
    // --------------------------------------------------------- softmax
    const int sw = warp - 4;
    const int h = sw / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const int64_t qrow = static_cast<int64_t>(qt) * kTile + r;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);
    float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
    float* lx = reinterpret_cast<float*>(smem + kOffLx);
    float* pdiag = reinterpret_cast<float*>(smem + kOffPdiag);
    const float C = p.score_scale_log2;
    const int ncols_o = h ? 72 : 64;  // O columns this half rescales (h=1 includes l at 128)
    const uint32_t col_o0 = kColO + (h ? 64u : 0u);
    const bool ragged = (N % kTile) != 0;
    float m_run = -INFINITY;
    bool my_abort = false;
    bool aborted = false;
    // all lanes poll; the outcome is made warp-uniform so tcgen05 .sync.aligned ops stay convergent
    auto wait_uniform = [&](int b, uint32_t parity) {
      bool ok = !my_abort && mbar_wait(bar(b), parity, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && !my_abort) {
        record_error(p.status, 4, abort_flag);
        my_abort = true;
      }
    };

    for (int j = 0; j < T; j++) {
      const int s = j & 1;
      float v[64];
      wait_uniform(kBarSFull + s, (j >> 1) & 1);
      tc_fence_after();
      if (!my_abort) {
        uint32_t rr[32];
        tmem_ld32(tl + kColS + s * kTile + 64 * h, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = __uint_as_float(rr[i]);
        tmem_ld32(tl + kColS + s * kTile + 64 * h + 32, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i++) v[32 + i] = __uint_as_float(rr[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; i++) v[i] = 0.0f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + s));

      const int64_t key0 = static_cast<int64_t>(j) * kTile + 64 * h;
      if (j == T - 1 && (p.causal || ragged)) {
#pragma unroll
        for (int i = 0; i < 64; i++) {
          const int64_t key = key0 + i;
          const bool valid = key < N && (!p.causal || key <= qrow);
          if (!valid) v[i] = -INFINITY;
        }
      }
      float bm[2];
#pragma unroll
      for (int b = 0; b < 2; b++) {
        float m0 = v[32 * b];
#pragma unroll
        for (int i = 1; i < 31; i += 2) m0 = fmax3(m0, v[32 * b + i], v[32 * b + i + 1]);
        bm[b] = fmaxf(m0, v[32 * b + 31]);
      }
      const float pm = fmaxf(bm[0], bm[1]);
      xchg[(s * 2 + h) * kTile + r] = pm;
      aborted = bar_red_or(1, 256, my_abort || *abort_flag);
      if (aborted) break;
      const float other = xchg[(s * 2 + (1 - h)) * kTile + r];
      const float m_new = fmax3(m_run, pm, other);
      const float mc = m_new * C;

      // P^ = Q*(exp(S/sqrt(d) - m_new)) per 32-key block, scale from the block maximum
      uint32_t words[8];
      uint32_t sbytes = 0;
#pragma unroll
      for (int b = 0; b < 2; b++) {
        uint32_t sbyte = 127;
        if (bm[b] == -INFINITY) {
#pragma unroll
          for (int g = 0; g < 4; g++) words[4 * b + g] = 0u;
        } else {
          const float xb = fmaf(bm[b], C, -mc);
          int e = static_cast<int>(ceilf(xb - kLog2Qmax));
          e = e < -127 ? -127 : e;
          const float off = mc + static_cast<float>(e);
#pragma unroll
          for (int g = 0; g < 4; g++) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; i++) y[i] = ex2_approx(fmaf(v[32 * b + 8 * g + i], C, -off));
            words[4 * b + g] = pack_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
          }
          sbyte = static_cast<uint32_t>(e + 127);
        }
        sbytes |= sbyte << (8 * b);
      }
      if (p.phat_codes != nullptr && qrow < N) {
        uint4* dst = reinterpret_cast<uint4*>(p.phat_codes + qrow * (static_cast<int64_t>(p.NT) * 64) +
                                              static_cast<int64_t>(bh) * N * p.NT * 64 + j * 64 + 32 * h);
        dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
        dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
        *reinterpret_cast<uint16_t*>(p.phat_scales + (static_cast<int64_t>(bh) * N + qrow) * p.NT * 4 + j * 4 +
                                     2 * h) = static_cast<uint16_t>(sbytes);
      }
      if (p.causal && j == qt && (quad >> 1) == h) {
        // the query's own 32-key block: keep P^ for the bf16-V product, drop it from the MMA operand
        const int lb = quad & 1;
        const float sc = __uint_as_float(((sbytes >> (8 * lb)) & 0xFFu) << 23);  // 2^(byte-127)
        float sum = 0.0f;
#pragma unroll
        for (int g = 0; g < 4; g++) {
          const uint32_t w = lb ? words[4 + g] : words[g];
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const float val = e2m1_decode((w >> (4 * i)) & 0xFu) * sc;
            pdiag[r * kPdiagStride + 8 * g + i] = val;
            sum += val;
          }
          if (lb) words[4 + g] = 0u; else words[g] = 0u;
        }
        lx[r] = sum;
      }
      if (j >= 2) wait_uniform(kBarPEmpty + s, ((j >> 1) - 1) & 1);
      {
        // P^ tile (128 rows x 64 bytes, 64-byte swizzle): this half owns 16-byte chunks 2h, 2h+1
        uint8_t* prow = smem + kOffP + s * kTileBytes + r * 64;
        const int x = (r >> 1) & 3;
        *reinterpret_cast<uint4*>(prow + (((2 * h) ^ x) << 4)) = make_uint4(words[0], words[1], words[2], words[3]);
        *reinterpret_cast<uint4*>(prow + (((2 * h + 1) ^ x) << 4)) = make_uint4(words[4], words[5], words[6], words[7]);
        *reinterpret_cast<uint16_t*>(smem + kOffPSF + s * kSfAtomBytes + (r % 32) * 16 + (r / 32) * 4 + 2 * h) =
            static_cast<uint16_t>(sbytes);
      }
      fence_proxy_async_smem();
      const float alpha = (j == 0) ? 0.0f : ex2_approx((m_run - m_new) * C);
      if (j >= 1) {
        wait_uniform(kBarODone, (j - 1) & 1);
        tc_fence_after();
        if (!my_abort && __any_sync(0xffffffffu, alpha != 1.0f)) {
          for (int c0 = 0; c0 < ncols_o; c0 += 8) {
            uint32_t o[8];
            tmem_ld8(tl + col_o0 + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st8(tl + col_o0 + c0, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + s));
      m_run = m_new;
    }

    // --------------------------------------------------------- epilogue
    if (!aborted) wait_uniform(kBarODone, (T - 1) & 1);
    tc_fence_after();
    __nv_bfloat16* vdiag = reinterpret_cast<__nv_bfloat16*>(smem + kOffVdiag);
    if (p.causal) {
      // bf16 V rows of the diagonal key tile (keys >= N read as 0)
      const int t = threadIdx.x - 128;
      const uint4* src = reinterpret_cast<const uint4*>(p.v_bf16 + (static_cast<int64_t>(bh) * N) * kD);
      for (int i = t; i < kTile * 16; i += 256) {
        const int row = i / 16;
        const int64_t key = static_cast<int64_t>(qt) * kTile + row;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (key < N) val = src[key * 16 + (i % 16)];
        reinterpret_cast<uint4*>(vdiag)[i] = val;
      }
    }
    if (h == 1) {
      float l = 0.0f;
      if (!my_abort && !aborted) {
        uint32_t o[8];
        tmem_ld8(tl + kColO + kD, o);
        tmem_wait_ld();
        l = __uint_as_float(o[0]);
      }
      if (p.causal) l += lx[r];
      lsum[r] = l;
    }
    named_bar_sync(2, 256);
    const float inv_l = 1.0f / lsum[r];
    if (!my_abort && !aborted) {
      float acc[64];
      uint32_t rr[32];
      tmem_ld32(tl + kColO + 64 * h, rr);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i++) acc[i] = __uint_as_float(rr[i]);
      tmem_ld32(tl + kColO + 64 * h + 32, rr);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i++) acc[32 + i] = __uint_as_float(rr[i]);
      if (p.causal) {
        const int kq = quad * 32;  // first key (within the diagonal tile) of this row's 32-token block
        for (int k = 0; k < 32; k++) {
          const float pk = pdiag[r * kPdiagStride + k];
          if (pk == 0.0f) continue;
          const __nv_bfloat162* vr = reinterpret_cast<const __nv_bfloat162*>(vdiag + (kq + k) * kD + 64 * h);
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const float2 f = __bfloat1622float2(vr[i]);
            acc[2 * i] = fmaf(pk, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(pk, f.y, acc[2 * i + 1]);
          }
        }
      }
      if (qrow < N) {
        float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(bh) * N + qrow) * kD + 64 * h);
#pragma unroll
        for (int i = 0; i < 16; i++)
          dst[i] = make_float4(acc[4 * i] * inv_l, acc[4 * i + 1] * inv_l, acc[4 * i + 2] * inv_l,
                               acc[4 * i + 3] * inv_l);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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
  Params p;
  p.q_scales = static_cast<const uint8_t*>(a.q_scales);
  p.k_scales = static_cast<const uint8_t*>(a.k_scales);
  p.v_scales = static_cast<const uint8_t*>(a.v_scales);
  p.v_bf16 = static_cast<const __nv_bfloat16*>(a.v_bf16);
  p.out = a.out;
  p.phat_codes = a.phat_codes;
  p.phat_scales = a.phat_scales;
  p.status = device_status_ptr();
  p.N = N;
  p.NT = static_cast<int>(NT);
  p.causal = a.causal;
  p.debug_flags = a.debug_flags;
  p.score_scale_log2 = kLog2e / 11.313708498984761f;  // log2(e) / sqrt(128)
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mxfp4_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(static_cast<unsigned>(NT), static_cast<unsigned>(BH));
  mxfp4_fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace mxattn
