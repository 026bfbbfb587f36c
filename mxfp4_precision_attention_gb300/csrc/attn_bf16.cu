// BF16 fused attention forward (comparison path for the MXFP4 kernel):
// the FlashAttention-2 recurrence of "MXAttention" Eqs. (2)-(8) with BF16
// operands, FP32 accumulation in TMEM, Bc = 128 key tiles.
//
//   S_j = Q K_j^T                 tcgen05.mma kind::f16 (bf16) -> TMEM
//   m   = max(m, rowmax S_j)      the 32-column maxima come with the TMEM load
//                                 (tcgen05.ld.red), masked last tiles from registers
//   P~  = exp(S_j/sqrt(d) - m)    fp32 in registers, rounded to bf16 -> TMEM
//   O   = diag(alpha) O + P V     tcgen05.mma kind::f16, P~ as the A operand
//                                 from TMEM, V as MN-major B from shared memory
//   l   = alpha l + sum P~        fp32 in the softmax thread (P~ before rounding,
//                                 as FlashAttention sums it)
//
// The structure is the MXFP4 kernel's: one CTA per pair of 128-row query
// tiles (A and B) of one head, streaming the head's K and V tiles once for
// both, with one S buffer in TMEM that the QK^T of one tile fills while the
// other tile's softmax warps work. Warp roles (12 warps): 0 TMA producer,
// 1 QK^T issuer, 2 P.V issuer and TMEM owner, 3 idle, 4-7 softmax of tile A,
// 8-11 of tile B, one full query row per thread (TMEM lane = row).
//   TMEM: S 128 | O_A 128 | O_B 128 | P_A 64 | P_B 64 (bf16 pairs) = 512 columns
//   shared memory: Q tiles 2 x 32 KB, K and V rings 2 x 32 KB each
//
// Queries and keys may differ in length (Nq, Nk); causal means key j is
// visible to query i iff j <= i. Every mbarrier wait is bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mxattn {
namespace {

constexpr uint32_t kHalfTile = 128 * 128;  // 64 bf16 x 128 rows (one 128B-swizzle column block)
constexpr uint32_t kTileB = 2 * kHalfTile;  // 32 KB
constexpr uint32_t kTmemCols = 512;

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr uint32_t kOffQ = 0;                          // 2 tiles
constexpr uint32_t kOffK = kOffQ + 2 * kTileB;        // kStages tiles
constexpr uint32_t kOffV = kOffK + kStages * kTileB;  // kStages tiles
constexpr uint32_t kOffBars = kOffV + kStages * kTileB;
constexpr int kNumBars = 24;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;
constexpr int kBarQFull = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kStages;
constexpr int kBarVFull = kBarKEmpty + kStages;
constexpr int kBarVEmpty = kBarVFull + kStages;
constexpr int kBarSFull = kBarVEmpty + kStages;  // [2 groups]
constexpr int kBarSEmpty = kBarSFull + 2;         // 4 arrivals
constexpr int kBarPFull = kBarSEmpty + 1;         // [2 groups], 4 arrivals
constexpr int kBarODone = kBarPFull + 2;          // [2 groups]
static_assert(kBarODone + 2 <= kNumBars, "barrier space");
constexpr uint32_t kColS = 0, kColO = 128, kColP = 384;

struct Params {
  float* out;
  int* status;
  int64_t Nq, Nk;  // query and key/value lengths
  int NTq, NTk;     // their 128-row tile counts
  int causal;
  uint32_t debug_flags;
  float score_scale_log2;
  int bh_major;  // grid x walks heads and y walks query-tile pairs (causal), else the reverse
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

// O += P V with P (M128 x K16 bf16) read from TMEM.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    bf16_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
  const int bh = static_cast<int>(p.bh_major ? blockIdx.x : blockIdx.y);
  const int slot = static_cast<int>(p.bh_major ? blockIdx.y : blockIdx.x);
  const int npairs = (p.NTq + 1) / 2;
  const int pair = p.causal ? (npairs - 1 - slot) : slot;  // causal: heaviest pairs first
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const bool has_b = qt1 < p.NTq;
  // causal: key j is visible to query i iff j <= i (both counted from 0)
  const int nt0 = p.causal ? (qt0 + 1 < p.NTk ? qt0 + 1 : p.NTk) : p.NTk;
  const int nt1 = has_b ? (p.causal ? (qt1 + 1 < p.NTk ? qt1 + 1 : p.NTk) : p.NTk) : 0;
  const int T = nt0 > nt1 ? nt0 : nt1;
  const int64_t Nq = p.Nq, Nk = p.Nk;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < kStages; s++) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int g = 0; g < 2; g++) {
      mbar_init(bar(kBarSFull + g), 1);
      mbar_init(bar(kBarPFull + g), 4);
      mbar_init(bar(kBarODone + g), 1);
    }
    mbar_init(bar(kBarSEmpty), 4);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_base_slot), kTmemCols);
    tmem_relinquish();
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
      const int ng = has_b ? 2 : 1;
      mbar_arrive_expect_tx(bar(kBarQFull), ng * kTileB);
      for (int g = 0; g < ng; g++) {
        const int qt = g ? qt1 : qt0;
        tma_load_3d(sb + kOffQ + g * kTileB, &tm_q, bar(kBarQFull), 0, qt * 128, bh);
        tma_load_3d(sb + kOffQ + g * kTileB + kHalfTile, &tm_q, bar(kBarQFull), 64, qt * 128, bh);
      }
      int nk = 0, nv = 0;
      for (int j = 0; j < T; j++) {
        const int st = j % kStages, u = j / kStages;
        if (u > 0 && !mbar_wait(bar(kBarKEmpty + st), (u - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + st), kTileB);
        tma_load_3d(sb + kOffK + st * kTileB, &tm_k, bar(kBarKFull + st), 0, j * 128, bh);
        tma_load_3d(sb + kOffK + st * kTileB + kHalfTile, &tm_k, bar(kBarKFull + st), 64, j * 128, bh);
        nk++;
        if (u > 0 && !mbar_wait(bar(kBarVEmpty + st), (u - 1) & 1, abort_flag)) {
          record_error(p.status, 4, abort_flag);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + st), kTileB);
        tma_load_3d(sb + kOffV + st * kTileB, &tm_v, bar(kBarVFull + st), 0, j * 128, bh);
        tma_load_3d(sb + kOffV + st * kTileB + kHalfTile, &tm_v, bar(kBarVFull + st), 64, j * 128, bh);
        nv++;
      }
      // every copy this thread issued must land before the CTA exits
      for (int j = (nk > kStages ? nk - kStages : 0); j < nk; j++)
        mbar_wait(bar(kBarKFull + j % kStages), (j / kStages) & 1, abort_flag);
      for (int j = (nv > kStages ? nv - kStages : 0); j < nv; j++)
        mbar_wait(bar(kBarVFull + j % kStages), (j / kStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- QK issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false);
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag);
      int n = 0;  // S productions so far
      for (int j = 0; ok && j < T; j++) {
        const int st = j % kStages;
        if (!mbar_wait(bar(kBarKFull + st), (j / kStages) & 1, abort_flag)) { ok = false; break; }
        const uint32_t ka = sb + kOffK + st * kTileB;
        for (int g = 0; g < 2; g++) {
          if (j >= (g ? nt1 : nt0)) continue;
          // the single S buffer is free once the previous production was read
          if (n >= 1 && !mbar_wait(bar(kBarSEmpty), (n - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t qa = sb + kOffQ + g * kTileB;
          for (int i = 0; i < 8; i++) {
            const uint32_t off = (i >> 2) * kHalfTile + (i & 3) * 32;
            mma_bf16(tmem + kColS, smem_desc(qa + off, 16, 1024, kSwizzle128B),
                     smem_desc(ka + off, 16, 1024, kSwizzle128B), id_s, i > 0 ? 1u : 0u);
          }
          if (!((p.debug_flags & kDebugNeverArriveS) && n == 0)) tc_commit(bar(kBarSFull + g));
          n++;
        }
        if (!ok) break;
        tc_commit(bar(kBarKEmpty + st));
      }
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  } else if (warp == 2) {
    // --------------------------------------------------------- PV issuer
    if (lane == 0) {
      const uint32_t id_o = idesc_bf16(128, 128, true);
      bool ok = true;
      for (int j = 0; ok && j < T; j++) {
        const int st = j % kStages;
        if (!mbar_wait(bar(kBarVFull + st), (j / kStages) & 1, abort_flag)) { ok = false; break; }
        const uint32_t va = sb + kOffV + st * kTileB;
        for (int g = 0; g < 2; g++) {
          if (j >= (g ? nt1 : nt0)) continue;
          if (!mbar_wait(bar(kBarPFull + g), j & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // K step i: keys 16i .. 16i+15, i.e. P columns 8i .. 8i+7 (two bf16 per column)
          for (int i = 0; i < 8; i++)
            mma_bf16_ta(tmem + kColO + 128 * g, tmem + kColP + 64 * g + 8 * i,
                        smem_desc(va + i * 2048, kHalfTile, 1024, kSwizzle128B), id_o, (j > 0 || i > 0) ? 1u : 0u);
          tc_commit(bar(kBarODone + g));
        }
        if (!ok) break;
        tc_commit(bar(kBarVEmpty + st));
      }
      if (!ok) record_error(p.status, 4, abort_flag);
    }
  } else if (warp >= 4) {
    // --------------------------------------------------------- softmax
    const int g = (warp - 4) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const int Tg = g ? nt1 : nt0;
    const int64_t qrow = static_cast<int64_t>(g ? qt1 : qt0) * 128 + r;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t ocol = kColO + 128 * g, pcol = kColP + 64 * g;
    const float C = p.score_scale_log2;
    const bool ragged = (Nk % 128) != 0;
    float m_run = -INFINITY, l_run = 0.0f;
    bool my_abort = false;
    auto wait_uniform = [&](int b, uint32_t parity) {
      bool ok = !my_abort && mbar_wait(bar(b), parity, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && !my_abort) {
        record_error(p.status, 4, abort_flag);
        my_abort = true;
      }
    };
    for (int j = 0; j < Tg && !my_abort; j++) {
      float v[128];
      float bm[4];
      wait_uniform(kBarSFull + g, j & 1);
      if (my_abort) break;
      tc_fence_after();
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32_max(tl + kColS, r0, bm[0]);
        tmem_ld32_max(tl + kColS + 32, r1, bm[1]);
        tmem_ld32_max(tl + kColS + 64, r2, bm[2]);
        tmem_ld32_max(tl + kColS + 96, r3, bm[3]);
        tmem_wait_ld();
        reg_fence32(r0);
        reg_fence32(r1);
        reg_fence32(r2);
        reg_fence32(r3);
#pragma unroll
        for (int b = 0; b < 4; b++) {
          uint32_t u = __float_as_uint(bm[b]);
          reg_fence1(u);
          bm[b] = __uint_as_float(u);
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
      float rowmax = fmax3(fmaxf(bm[0], bm[1]), bm[2], bm[3]);
      if (j == Tg - 1 && (p.causal || ragged)) {
        // the last tile's masked keys are -inf in v only: its maximum comes from v
        const int64_t key0 = static_cast<int64_t>(j) * 128;
#pragma unroll
        for (int i = 0; i < 128; i++) {
          const int64_t key = key0 + i;
          if (!(key < Nk && (!p.causal || key <= qrow))) v[i] = -INFINITY;
        }
        rowmax = v[0];
#pragma unroll
        for (int i = 1; i < 127; i += 2) rowmax = fmax3(rowmax, v[i], v[i + 1]);
        rowmax = fmaxf(rowmax, v[127]);
      }
      const float m_new = fmaxf(m_run, rowmax);
      const float mc = m_new * C;
      const float alpha = (j == 0) ? 0.0f : ex2_approx((m_run - m_new) * C);
      uint32_t packed[64];
      float2 sum2 = make_float2(0.0f, 0.0f);
      const float2 c2 = make_float2(C, C), nmc2 = make_float2(-mc, -mc);
#pragma unroll
      for (int i = 0; i < 64; i++) {
        const float2 x = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), c2, nmc2);
        const float e0 = ex2_approx(x.x), e1 = ex2_approx(x.y);
        packed[i] = pack_bf16x2(e0, e1);
        sum2 = __fadd2_rn(sum2, make_float2(e0, e1));
      }
      l_run = fmaf(alpha, l_run, sum2.x + sum2.y);
      if (j >= 1) {
        // P.V of tile j-1 is complete: this group's P buffer is free and O is stable
        wait_uniform(kBarODone + g, (j - 1) & 1);
        if (my_abort) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
          for (int c = 0; c < 4; c++) {
            uint32_t o[32];
            tmem_ld32(tl + ocol + 32 * c, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 y = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
              o[i] = __float_as_uint(y.x);
              o[i + 1] = __float_as_uint(y.y);
            }
            tmem_st32(tl + ocol + 32 * c, o);
          }
        }
      }
      {
        uint32_t w0[32], w1[32];
#pragma unroll
        for (int i = 0; i < 32; i++) {
          w0[i] = packed[i];
          w1[i] = packed[32 + i];
        }
        tmem_st32(tl + pcol, w0);
        tmem_st32(tl + pcol + 32, w1);
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
        const float inv_l = 1.0f / l_run;
        float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(bh) * Nq + qrow) * kD);
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
          uint32_t o[32];
          tmem_ld32(tl + ocol + 32 * c, o);  // warp-wide; rows past Nq load but do not store
          tmem_wait_ld();
          reg_fence32(o);
          if (qrow < Nq) {
#pragma unroll
            for (int i = 0; i < 8; i++)
              dst[8 * c + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                           __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_bf16_forward(const Bf16FwdArgs& a, cudaStream_t s) {
  const int64_t Nq = a.Nq, Nk = a.Nk, BH = a.BH;
  const int64_t NTq = ceil_div(Nq, 128), NTk = ceil_div(Nk, 128);
  alignas(64) CUtensorMap tq, tk, tv;
  const uint64_t dq[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Nq), static_cast<uint64_t>(BH)};
  const uint64_t sq[2] = {kD * 2, static_cast<uint64_t>(Nq) * kD * 2};
  const uint64_t dk[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Nk), static_cast<uint64_t>(BH)};
  const uint64_t sk[2] = {kD * 2, static_cast<uint64_t>(Nk) * kD * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (!encode_tensor_map(&tq, 1, 3, const_cast<void*>(a.q), dq, sq, box, 128)) return cudaErrorInvalidValue;
  if (!encode_tensor_map(&tk, 1, 3, const_cast<void*>(a.k), dk, sk, box, 128)) return cudaErrorInvalidValue;
  if (!encode_tensor_map(&tv, 1, 3, const_cast<void*>(a.v), dk, sk, box, 128)) return cudaErrorInvalidValue;
  Params p;
  p.out = a.out;
  p.status = device_status_ptr();
  p.Nq = Nq;
  p.Nk = Nk;
  p.NTq = static_cast<int>(NTq);
  p.NTk = static_cast<int>(NTk);
  p.causal = a.causal;
  p.debug_flags = a.debug_flags;
  p.score_scale_log2 = 1.4426950408889634f / 11.313708498984761f;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(bf16_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // causal: heads on x so that every head's longest query-tile pair starts first
  const int64_t npairs = (NTq + 1) / 2;
  p.bh_major = (a.causal && npairs <= 65535) ? 1 : 0;
  dim3 grid = p.bh_major ? dim3(static_cast<unsigned>(BH), static_cast<unsigned>(npairs))
                         : dim3(static_cast<unsigned>(npairs), static_cast<unsigned>(BH));
  bf16_fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace mxattn
