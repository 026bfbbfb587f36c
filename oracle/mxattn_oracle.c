/*
 * MXAttention CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 restatement of what the MXAttention forward pass
 * computes, written from "MXAttention: Data-Free Optimal Scaling and
 * Pre-Normalization Quantization for MXFP4 Attention" (arXiv 2607.24377) and
 * the MatX note "leaky quantization" (causal section). Only the test-suite,
 * the smoke check and the benchmark's CPU-baseline leg may load this file; the
 * product path never does. It shares no code, header, table or constant with
 * the CUDA kernels.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   R1  E2M1 projection: round to nearest, ties to the even code (the code
 *       whose mantissa bit is 0), saturating at +-6. The sign of the input is
 *       kept, so a negative value that rounds to zero yields code 0x8.
 *   R2  Hadamard rotation: Sylvester H_128 in natural order, R_H = H/sqrt(128),
 *       evaluated in binary32 as seven butterfly stages h = 1,2,...,64 where
 *       each pair (i, i+h), i&h == 0, becomes (a+b, a-b), followed by one
 *       multiply with the binary32 value nearest 2^-3.5.
 *   R3  UOS exponent e = ceil(log2(M/7.25)) is evaluated exactly through
 *       frexp, then clamped to the E8M0 range [-127, 127]; it is stored as the
 *       biased byte e+127. An all-zero block gets sigma = 1 (byte 127).
 *   R4  Blocks: Q/K per token over channels [32b, 32b+32); V per channel over
 *       tokens [32t, 32t+32) (last block short); P~ per query row over keys
 *       [32t, 32t+32) counted from key 0.
 *   R5  Online softmax with fixed key tiles of Bc = 128 in increasing key order.
 *   R6  Causal: keys j > i are masked before the row maximum; for the 32-token
 *       V block that holds the query itself, P^ multiplies the unquantized
 *       (bf16) V rows instead of V^, so no later token can reach row i.
 *
 * NVFP4 comparison format (section 1: E2M1 values in 16-element blocks with
 * an E4M3 block scale and a tensor-level scale; section 5.2: the direct NVFP4
 * baseline quantizes Q, K, V and P~ for the two products, with no smoothing
 * and no softmax-path scaling):
 *   N1  E4M3 block scales: round to nearest, ties to the even code, values at
 *       or above 448 saturate to 448 (the largest finite E4M3 value).
 *   N2  A block's scale maps its maximum |x| to the E2M1 maximum 6.
 *   N3  Tensor scale of Q, K, V: encode factor e_t = 2688 / amax over the
 *       whole tensor (2688 = 6 * 448), so the largest block scale is 448;
 *       e_t = 1 if the tensor is all zero. P~ has no tensor scale (e_t = 1).
 *   N4  Binary32 order of operations (the GPU quantizers use the same):
 *         e_t = fl(2688 / amax)
 *         sc  = E4M3(fl(fl(M / 6) * e_t)), S = value of sc
 *         sc == 0: every code 0; else k = fl(e_t / S), code = E2M1(fl(x * k))
 *       dequantized value = E2M1 value * S / e_t.
 *   N5  Blocks of 16: Q/K per token over channels [16b, 16b+16), V per
 *       channel over tokens [16t, 16t+16), P~ per row over keys [16t, 16t+16).
 *       Causal: the query's own 16-token V block uses the bf16 V rows (R6).
 *   N6  Q and K are not rotated.
 *
 * Row-sum diagnostic of a quantized materialized P (section 5.5.2, Fig. 7 B):
 *   D1  Each row of P is quantized in blocks of 32 consecutive keys counted
 *       from key 0 (R4), with the block quantizer of Algorithm 1 under the
 *       given scale rule. The row-sum error sum(Q(P) - P) is split by the
 *       outcome of each element with P > 0: zeroing (Q(P) = 0), saturation
 *       (P / 2^e above the largest E2M1 value 6, so Q(P) = 6 * 2^e),
 *       downward rounding (any other Q(P) < P) and upward rounding
 *       (Q(P) > P). The four parts sum to the whole error.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared [-fopenmp] -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_D 128
#define ORC_BLOCK 32

/* ------------------------------------------------------------------ E2M1
 * Nonnegative E2M1 grid, Eq. (9)/(20); code index = magnitude bits.        */
static const double kGrid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code) {
  double m = kGrid[code & 7];
  return (code & 8) ? -m : m;
}

/* Round-to-nearest projection onto the finite E2M1 grid with saturation at
 * +-6 (Eq. 10), ties to the even code (reading R1). Returns the 4-bit code. */
int orc_e2m1_code(double v) {
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  if (a >= 6.0) return 7 | (neg << 3); /* out of range: saturate at +-6 (Eq. 10) */
  int best = 0;
  double bestd = fabs(a - kGrid[0]);
  for (int c = 1; c < 8; c++) {
    double d = fabs(a - kGrid[c]);
    if (d < bestd || (d == bestd && (c % 2) == 0 && (best % 2) != 0)) {
      best = c;
      bestd = d;
    }
  }
  return best | (neg << 3);
}

/* --------------------------------------------------------- scale rules
 * rule 0: UOS, e = ceil(log2(M / 7.25))           (Eq. 13 / 19, Alg. 1)
 * rule 1: OCP, e = floor(log2 M) - 2              (Eq. 11 / 97)
 * rule 2: TFS, e = ceil(log2(M / 6))              (Eq. 14)
 * rule 3: e = ceil(log2(M / q)) for a given q in (4, 8]: the Q_max sweep of
 *         section 5.5.1 (q = 7.25 is UOS, q = 6 is TFS)
 * M > 0. With M = f * 2^E, f in [0.5, 1):
 *   ceil(log2(M/q)) = E - 3 if f <= q/8 else E - 2, for q in (4, 8]
 *   (and E - 4 if f <= q/16, which needs q = 8 and f = 1/2);
 *   floor(log2 M)   = E - 1.
 * Result clamped to the E8M0 exponent range [-127, 127].                   */
double orc_uos_qmax(void) { return 7.25; }

int orc_scale_exponent_q(double M, int rule, double qmax) {
  int E;
  double f = frexp(M, &E);
  int e;
  if (rule == 1) {
    e = (E - 1) - 2;
  } else {
    double q = (rule == 2) ? 6.0 : (rule == 3 ? qmax : orc_uos_qmax());
    /* smallest e with M / 2^e <= q; f <= q/16 happens only for q = 8, f = 1/2 */
    e = (f <= q / 16.0) ? E - 4 : ((f <= q / 8.0) ? E - 3 : E - 2);
  }
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

int orc_scale_exponent(double M, int rule) { return orc_scale_exponent_q(M, rule, 7.25); }

/* Quantize one block of n values (Algorithm 1). codes[i] receives the 4-bit
 * code, the return value is the biased E8M0 byte.                          */
static int quantize_block(const double* v, int n, int rule, double q, uint8_t* codes) {
  double M = 0.0;
  for (int i = 0; i < n; i++) {
    double a = fabs(v[i]);
    if (a > M) M = a;
  }
  if (M == 0.0) { /* all-zero block: sigma = 1, every element 0 */
    for (int i = 0; i < n; i++) codes[i] = 0;
    return 127;
  }
  int e = orc_scale_exponent_q(M, rule, q);
  for (int i = 0; i < n; i++) codes[i] = (uint8_t)orc_e2m1_code(ldexp(v[i], -e));
  return e + 127;
}

/* Dequantized value of one block element: code value times 2^(byte-127). */
static double dq(uint8_t code, uint8_t sbyte) { return ldexp(orc_e2m1_value(code), (int)sbyte - 127); }

/* --------------------------------------------------------------- bf16 */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------- E4M3 (N1)
 * Finite nonnegative E4M3 codes 0..126 (0x7F is NaN): exponent field
 * c >> 3, mantissa c & 7; field 0 is subnormal (m/8 * 2^-6), else
 * (1 + m/8) * 2^(field - 7). Largest finite value: code 126 = 448.          */
double orc_e4m3_value(int code) {
  const int ef = (code >> 3) & 15, m = code & 7;
  if (ef == 0) return ldexp((double)m, -9);
  return ldexp(8.0 + m, ef - 10);
}

/* Nearest finite E4M3 code to v >= 0, ties to the even code; >= 448 -> 126. */
int orc_e4m3_code(double v) {
  if (!(v < 448.0)) return 126;
  int best = 0;
  double bestd = fabs(v);
  for (int c = 1; c <= 126; c++) {
    const double d = fabs(v - orc_e4m3_value(c));
    if (d < bestd || (d == bestd && (c % 2) == 0 && (best % 2) != 0)) {
      best = c;
      bestd = d;
    }
  }
  return best;
}

/* Tensor encode factor e_t (N3, N4). */
float orc_nvfp4_encode(float amax) { return amax > 0.0f ? 2688.0f / amax : 1.0f; }

/* Quantize one block of n binary32 values with encode factor e_t (N2, N4).
 * codes[i] receives the 4-bit code; returns the E4M3 scale byte.           */
static int nv_block(const float* x, int n, float e_t, uint8_t* codes) {
  float M = 0.0f;
  for (int i = 0; i < n; i++)
    if (fabsf(x[i]) > M) M = fabsf(x[i]);
  const float t = M / 6.0f;
  const float v = t * e_t;
  const int sc = orc_e4m3_code((double)v);
  const float S = (float)orc_e4m3_value(sc);
  if (sc == 0) {
    for (int i = 0; i < n; i++) codes[i] = 0;
    return 0;
  }
  const float k = e_t / S;
  for (int i = 0; i < n; i++) {
    const float y = x[i] * k;
    codes[i] = (uint8_t)orc_e2m1_code((double)y);
  }
  return sc;
}

/* Dequantized NVFP4 element: E2M1 value * S / e_t, in float64. */
static double nv_dq(uint8_t code, uint8_t sc, float e_t) {
  return orc_e2m1_value(code) * orc_e4m3_value(sc) / (double)e_t;
}

/* ------------------------------------------------------ Hadamard (R2)
 * y = x R_H with R_H = H_128 / sqrt(128), Sylvester order. Binary32.       */
void orc_hadamard_fp32(const uint16_t* x_bf16, float* y) {
  float z[ORC_D];
  for (int i = 0; i < ORC_D; i++) z[i] = bf16_to_f32(x_bf16[i]);
  for (int h = 1; h < ORC_D; h <<= 1) {
    for (int i = 0; i < ORC_D; i++) {
      if (i & h) continue;
      float a = z[i], b = z[i + h];
      float s = a + b;
      float d = a - b;
      z[i] = s;
      z[i + h] = d;
    }
  }
  const float inv_sqrt_d = (float)0.08838834764831845; /* nearest binary32 to 2^-3.5 */
  for (int i = 0; i < ORC_D; i++) y[i] = z[i] * inv_sqrt_d;
}

/* ------------------------------------------------- Q / K quantization
 * Algorithm 2 (section 4.3), Q/K steps: rotate each token, then quantize each 32-channel block.
 * codes: rows x 128 (one code per byte); scales: rows x 4 biased bytes.    */
void orc_rotate_quantize_qk(const uint16_t* x, int64_t rows, int rule, double q, int rotate, uint8_t* codes,
                            uint8_t* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    float y[ORC_D];
    if (rotate) {
      orc_hadamard_fp32(x + r * ORC_D, y);
    } else {
      for (int i = 0; i < ORC_D; i++) y[i] = bf16_to_f32(x[r * ORC_D + i]);
    }
    for (int b = 0; b < ORC_D / ORC_BLOCK; b++) {
      double v[ORC_BLOCK];
      for (int i = 0; i < ORC_BLOCK; i++) v[i] = (double)y[b * ORC_BLOCK + i];
      scales[r * 4 + b] = (uint8_t)quantize_block(v, ORC_BLOCK, rule, q, codes + r * ORC_D + b * ORC_BLOCK);
    }
  }
}

/* ---------------------------------------------------- V quantization
 * Algorithm 2 (section 4.3), V step, with token blocks (R4). v: [BH][N][128] bf16.
 * codes: [BH][N][128] (token-major, one code per byte);
 * scales: [BH][128][nblk], nblk = ceil(N/32).                              */
void orc_quantize_v(const uint16_t* v, int64_t BH, int64_t N, int rule, double q, uint8_t* codes, uint8_t* scales) {
  const int64_t nblk = (N + ORC_BLOCK - 1) / ORC_BLOCK;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bh = 0; bh < BH; bh++) {
    for (int64_t c = 0; c < ORC_D; c++) {
      for (int64_t t = 0; t < nblk; t++) {
        int64_t n0 = t * ORC_BLOCK, n1 = n0 + ORC_BLOCK < N ? n0 + ORC_BLOCK : N;
        int n = (int)(n1 - n0);
        double vals[ORC_BLOCK];
        uint8_t cb[ORC_BLOCK];
        for (int i = 0; i < n; i++) vals[i] = (double)bf16_to_f32(v[((bh * N) + n0 + i) * ORC_D + c]);
        scales[(bh * ORC_D + c) * nblk + t] = (uint8_t)quantize_block(vals, n, rule, q, cb);
        for (int i = 0; i < n; i++) codes[((bh * N) + n0 + i) * ORC_D + c] = cb[i];
      }
    }
  }
}

/* ------------------------------------------- NVFP4 Q/K and V (N1-N6)
 * Q/K: x [rows][128] bf16; codes [rows][128] one per byte; scales [rows][8]
 * E4M3 bytes (16-channel blocks); *e_t: the tensor's encode factor.         */
void orc_nvfp4_quantize_qk(const uint16_t* x, int64_t rows, uint8_t* codes, uint8_t* scales, float* e_t) {
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * ORC_D; i++) {
    const float a = fabsf(bf16_to_f32(x[i]));
    if (a > amax) amax = a;
  }
  const float et = orc_nvfp4_encode(amax);
  *e_t = et;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    float v[ORC_D];
    for (int c = 0; c < ORC_D; c++) v[c] = bf16_to_f32(x[r * ORC_D + c]);
    for (int b = 0; b < ORC_D / 16; b++) scales[r * 8 + b] = (uint8_t)nv_block(v + 16 * b, 16, et, codes + r * ORC_D + 16 * b);
  }
}

/* V: v [BH][N][128] bf16; codes [BH][N][128]; scales [BH][128][ceil(N/16)]
 * (16-token blocks per channel, the last one short); *e_t as above.        */
void orc_nvfp4_quantize_v(const uint16_t* v, int64_t BH, int64_t N, uint8_t* codes, uint8_t* scales, float* e_t) {
  float amax = 0.0f;
  for (int64_t i = 0; i < BH * N * ORC_D; i++) {
    const float a = fabsf(bf16_to_f32(v[i]));
    if (a > amax) amax = a;
  }
  const float et = orc_nvfp4_encode(amax);
  *e_t = et;
  const int64_t nblk = (N + 15) / 16;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bh = 0; bh < BH; bh++) {
    for (int c = 0; c < ORC_D; c++) {
      for (int64_t t = 0; t < nblk; t++) {
        const int64_t n0 = t * 16;
        const int n = (int)(N - n0 < 16 ? N - n0 : 16);
        float vals[16];
        uint8_t cb[16];
        for (int i = 0; i < n; i++) vals[i] = bf16_to_f32(v[(bh * N + n0 + i) * ORC_D + c]);
        scales[(bh * ORC_D + c) * nblk + t] = (uint8_t)nv_block(vals, n, et, cb);
        for (int i = 0; i < n; i++) codes[(bh * N + n0 + i) * ORC_D + c] = cb[i];
      }
    }
  }
}

/* ------------------------------------------------ online softmax core
 * Algorithm 2 (section 4.3) loop, Eqs. 2-8 with PNQ (Eqs. 44-48), for one query row against one head's keys, float64.
 *   q      : 128 query values (already dequantized)
 *   K, V   : N x 128 key / value values (already dequantized)
 *   Vraw   : N x 128 unquantized values, used on the causal diagonal block
 *   i      : the query's token index (causal masking and the diagonal block)
 * causal: 0 = none; 1 = keys j > i masked and the query's own 32-token V block
 * taken unquantized from Vraw (the reading that removes the leak the MatX note
 * describes); 2 = the same mask, with that block re-quantized per channel over
 * tokens b0..i only (tokens after i left out of the block maximum), using the
 * P~ rule p_rule / p_q.
 * Options: quant_p (PNQ quantizer on), placement (0 = PNQ: l from P^,
 * 1 = direct: l from P~, Eq. 16-17), p_rule (scale rule for P~), bc (tile),
 * nv (P~ as NVFP4: 16-key blocks with the E4M3 scale of M/6, and the
 * causal diagonal block is the query's own 16-token V block).
 * Outputs: o[128], *ell; optional phat[ntiles*bc] (P^ of each tile before any
 * later rescale, masked slots 0) and mhist[ntiles] (running max after each
 * tile).                                                                    */
typedef struct {
  int causal;
  int quant_p;
  int placement;
  int p_rule;
  int bc;
  double p_q;
  int nv; /* 1: P~ quantized as NVFP4 (16-key blocks, E4M3 scale of M/6, N1-N5) */
  const double* phat_in; /* replay: this row's P^ per tile (ntiles*bc) given, not computed */
} orc_opts;

static void online_softmax_row(const double* q, const double* K, const double* V, const double* Vraw,
                               int64_t N, int64_t i, const orc_opts* op, double* o, double* ell_out,
                               double* phat, double* mhist) {
  const int bc = op->bc;
  const double inv_sqrt_d = 1.0 / sqrt((double)ORC_D);
  int64_t ntiles = (N + bc - 1) / bc;
  if (op->causal) ntiles = i / bc + 1;
  double m = -INFINITY, ell = 0.0;
  double acc[ORC_D];
  for (int c = 0; c < ORC_D; c++) acc[c] = 0.0;
  double* S = (double*)malloc(sizeof(double) * bc);
  double* Pt = (double*)malloc(sizeof(double) * bc);
  double* Ph = (double*)malloc(sizeof(double) * bc);
  unsigned char* valid = (unsigned char*)malloc(bc);
  /* causal == 2: the diagonal V block, re-quantized over tokens b0..i */
  const int64_t b0 = (i / ORC_BLOCK) * ORC_BLOCK;
  const int npre = (int)(i - b0 + 1);
  double* Vd = NULL;
  if (op->causal == 2) {
    Vd = (double*)malloc(sizeof(double) * ORC_BLOCK * ORC_D);
    for (int c = 0; c < ORC_D; c++) {
      double vals[ORC_BLOCK];
      uint8_t cb[ORC_BLOCK];
      for (int t = 0; t < npre; t++) vals[t] = Vraw[(b0 + t) * ORC_D + c];
      int sb = quantize_block(vals, npre, op->p_rule, op->p_q, cb);
      for (int t = 0; t < npre; t++) Vd[t * ORC_D + c] = dq(cb[t], (uint8_t)sb);
    }
  }
  for (int64_t j = 0; j < ntiles; j++) {
    const int64_t k0 = j * bc;
    /* Eq. 2: S = Q^ K^T / sqrt(d) */
    double rowmax = -INFINITY;
    for (int kk = 0; kk < bc; kk++) {
      int64_t key = k0 + kk;
      valid[kk] = (key < N) && (!op->causal || key <= i);
      if (!valid[kk]) {
        S[kk] = -INFINITY;
        continue;
      }
      double dot = 0.0;
      for (int c = 0; c < ORC_D; c++) dot += q[c] * K[key * ORC_D + c];
      S[kk] = dot * inv_sqrt_d;
      if (S[kk] > rowmax) rowmax = S[kk];
    }
    /* Eqs. 3-4: running max and alpha */
    double m_new = m > rowmax ? m : rowmax;
    double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    /* Eq. 5: P~ = exp(S - m_new) */
    for (int kk = 0; kk < bc; kk++) Pt[kk] = valid[kk] ? exp(S[kk] - m_new) : 0.0;
    /* Eq. 44: P^ = Q*(P~), 32-key blocks counted from key 0 (16 for NVFP4) */
    const int pblk = op->nv ? 16 : ORC_BLOCK;
    for (int b0 = 0; b0 < bc; b0 += pblk) {
      if (op->phat_in) {
        /* replay: the given P^ (a kernel's dumped codes and scales) on the valid keys */
        for (int t = 0; t < pblk; t++) Ph[b0 + t] = valid[b0 + t] ? op->phat_in[j * bc + b0 + t] : 0.0;
      } else if (op->quant_p && op->nv) {
        /* N2, N4 with e_t = 1, in float64: S = E4M3(fl(M / 6)), code = E2M1(P~ / S) */
        double M = 0.0;
        for (int t = 0; t < 16; t++)
          if (Pt[b0 + t] > M) M = Pt[b0 + t];
        const int sc = orc_e4m3_code((double)(float)(M / 6.0));
        const double S = orc_e4m3_value(sc);
        for (int t = 0; t < 16; t++)
          Ph[b0 + t] = sc == 0 ? 0.0 : orc_e2m1_value(orc_e2m1_code(Pt[b0 + t] / S)) * S;
      } else if (op->quant_p) {
        uint8_t cb[ORC_BLOCK];
        int sb = quantize_block(Pt + b0, ORC_BLOCK, op->p_rule, op->p_q, cb);
        for (int t = 0; t < ORC_BLOCK; t++) Ph[b0 + t] = dq(cb[t], (uint8_t)sb);
      } else {
        for (int t = 0; t < pblk; t++) Ph[b0 + t] = Pt[b0 + t];
      }
    }
    /* Eq. 47 (PNQ) or Eq. 16 (direct placement) */
    double tile_sum = 0.0;
    for (int kk = 0; kk < bc; kk++) tile_sum += (op->placement == 0) ? Ph[kk] : Pt[kk];
    ell = alpha * ell + tile_sum;
    /* Eq. 48: O = diag(alpha) O + P^ V^_j -- the tile product P^ V^_j first,
     * then the update, as l = alpha l + sum P^ above */
    double tp[ORC_D];
    for (int c = 0; c < ORC_D; c++) tp[c] = 0.0;
    for (int kk = 0; kk < bc; kk++) {
      if (!valid[kk] || Ph[kk] == 0.0) continue;
      int64_t key = k0 + kk;
      const int vblk = op->nv ? 16 : ORC_BLOCK;
      const int diag = op->causal && (key / vblk) == (i / vblk);
      const double* vrow = !diag ? V + key * ORC_D : (op->causal == 2 ? Vd + (key - b0) * ORC_D : Vraw + key * ORC_D);
      for (int c = 0; c < ORC_D; c++) tp[c] += Ph[kk] * vrow[c];
    }
    for (int c = 0; c < ORC_D; c++) acc[c] = alpha * acc[c] + tp[c];
    m = m_new;
    if (phat) memcpy(phat + j * bc, Ph, sizeof(double) * bc);
    if (mhist) mhist[j] = m;
  }
  /* Eq. 8: O = diag(l)^-1 O */
  for (int c = 0; c < ORC_D; c++) o[c] = acc[c] / ell;
  *ell_out = ell;
  free(Vd);
  free(S);
  free(Pt);
  free(Ph);
  free(valid);
}

/* Entry on real-valued inputs (used by the oracle's own pins).
 * q_rows: nrows x 128 query values; row_tok: token index of each query row.
 * K, V, Vraw: N x 128 (Vraw may be NULL when not causal).                   */
void orc_online_softmax(const double* q_rows, const int64_t* row_tok, int64_t nrows, const double* K,
                        const double* V, const double* Vraw, int64_t N, int causal, int quant_p,
                        int placement, int p_rule, double p_q, int bc, double* out, double* ell, double* phat,
                        double* mhist) {
  orc_opts op = {causal, quant_p, placement, p_rule, bc, p_q, 0, NULL};
  const int64_t ntiles = (N + bc - 1) / bc;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; r++) {
    online_softmax_row(q_rows + r * ORC_D, K, V, Vraw ? Vraw : V, N, row_tok[r], &op, out + r * ORC_D,
                       ell + r, phat ? phat + r * ntiles * bc : NULL, mhist ? mhist + r * ntiles : NULL);
  }
}

/* ------------------------------------------------------ full forward
 * Alg. 2 on quantized tensors. Inputs in the oracle's logical layouts:
 *   qc, kc, vc : [BH][N][128] codes, one per byte
 *   qs, ks     : [BH][N][4] biased scale bytes (per token, per channel block)
 *   vs         : [BH][128][nblk] biased scale bytes (per channel, per token block)
 *   vraw       : [BH][N][128] bf16 values of V (causal diagonal blocks), or NULL
 * rows: nrows pairs (bh, token). Outputs as in orc_online_softmax.
 * Rows are grouped by head by the caller for efficiency (not required).     */
int orc_forward(const uint8_t* qc, const uint8_t* qs, const uint8_t* kc, const uint8_t* ks, const uint8_t* vc,
                const uint8_t* vs, const uint16_t* vraw, int64_t BH, int64_t N, int causal, int placement,
                int p_rule, double p_q, int quant_p, int bc, const int64_t* rows, int64_t nrows, double* out,
                double* ell, double* phat, double* mhist) {
  if (bc <= 0 || bc % ORC_BLOCK != 0) return 1;
  const int64_t nblk = (N + ORC_BLOCK - 1) / ORC_BLOCK;
  const int64_t ntiles = (N + bc - 1) / bc;
  orc_opts op = {causal, quant_p, placement, p_rule, bc, p_q, 0, NULL};
  double* K = (double*)malloc(sizeof(double) * N * ORC_D);
  double* V = (double*)malloc(sizeof(double) * N * ORC_D);
  double* Vr = (double*)malloc(sizeof(double) * N * ORC_D);
  if (!K || !V || !Vr) {
    free(K);
    free(V);
    free(Vr);
    return 2;
  }
  for (int64_t bh = 0; bh < BH; bh++) {
    int any = 0;
    for (int64_t r = 0; r < nrows; r++) any |= (rows[2 * r] == bh);
    if (!any) continue;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
      for (int c = 0; c < ORC_D; c++) {
        const int64_t e = (bh * N + n) * ORC_D + c;
        K[n * ORC_D + c] = dq(kc[e], ks[(bh * N + n) * 4 + c / ORC_BLOCK]);
        V[n * ORC_D + c] = dq(vc[e], vs[(bh * ORC_D + c) * nblk + n / ORC_BLOCK]);
        Vr[n * ORC_D + c] = vraw ? (double)bf16_to_f32(vraw[e]) : V[n * ORC_D + c];
      }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; r++) {
      if (rows[2 * r] != bh) continue;
      const int64_t i = rows[2 * r + 1];
      double q[ORC_D];
      for (int c = 0; c < ORC_D; c++) {
        const int64_t e = (bh * N + i) * ORC_D + c;
        q[c] = dq(qc[e], qs[(bh * N + i) * 4 + c / ORC_BLOCK]);
      }
      online_softmax_row(q, K, V, Vr, N, i, &op, out + r * ORC_D, ell + r,
                         phat ? phat + r * ntiles * bc : NULL, mhist ? mhist + r * ntiles : NULL);
    }
  }
  free(K);
  free(V);
  free(Vr);
  return 0;
}

/* ------------------------------------------------ NVFP4 forward (N1-N6)
 * The same loop with NVFP4 operands: qc, kc, vc [BH][N][128] codes; qs, ks
 * [BH][N][8] E4M3 bytes; vs [BH][128][ceil(N/16)]; q_et, k_et, v_et the
 * tensors' encode factors. causal 0 or 1 (the own 16-token V block on bf16).
 * P~ is NVFP4-quantized when quant_p (N2, N4 with e_t = 1). phat_in (or NULL):
 * replay mode, row r's P^ for every tile given ([nrows][ntiles*128]), so a
 * kernel's own P^ decisions can be replayed through the float64 loop.      */
int orc_forward_nvfp4(const uint8_t* qc, const uint8_t* qs, float q_et, const uint8_t* kc, const uint8_t* ks,
                      float k_et, const uint8_t* vc, const uint8_t* vs, float v_et, const uint16_t* vraw, int64_t BH,
                      int64_t N, int causal, int placement, int quant_p, const int64_t* rows, int64_t nrows,
                      double* out, double* ell, double* phat, double* mhist, const double* phat_in) {
  if (causal != 0 && causal != 1) return 1;
  const int bc = 128;
  const int64_t nblk = (N + 15) / 16;
  const int64_t ntiles = (N + bc - 1) / bc;
  const orc_opts op0 = {causal, quant_p, placement, 0, bc, 7.25, 1, NULL};
  double* K = (double*)malloc(sizeof(double) * N * ORC_D);
  double* V = (double*)malloc(sizeof(double) * N * ORC_D);
  double* Vr = (double*)malloc(sizeof(double) * N * ORC_D);
  if (!K || !V || !Vr) {
    free(K);
    free(V);
    free(Vr);
    return 2;
  }
  for (int64_t bh = 0; bh < BH; bh++) {
    int any = 0;
    for (int64_t r = 0; r < nrows; r++) any |= (rows[2 * r] == bh);
    if (!any) continue;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
      for (int c = 0; c < ORC_D; c++) {
        const int64_t e = (bh * N + n) * ORC_D + c;
        K[n * ORC_D + c] = nv_dq(kc[e], ks[(bh * N + n) * 8 + c / 16], k_et);
        V[n * ORC_D + c] = nv_dq(vc[e], vs[(bh * ORC_D + c) * nblk + n / 16], v_et);
        Vr[n * ORC_D + c] = vraw ? (double)bf16_to_f32(vraw[e]) : V[n * ORC_D + c];
      }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; r++) {
      if (rows[2 * r] != bh) continue;
      const int64_t i = rows[2 * r + 1];
      double q[ORC_D];
      for (int c = 0; c < ORC_D; c++) {
        const int64_t e = (bh * N + i) * ORC_D + c;
        q[c] = nv_dq(qc[e], qs[(bh * N + i) * 8 + c / 16], q_et);
      }
      orc_opts op = op0;
      op.phat_in = phat_in ? phat_in + r * ntiles * bc : NULL;
      online_softmax_row(q, K, V, Vr, N, i, &op, out + r * ORC_D, ell + r,
                         phat ? phat + r * ntiles * bc : NULL, mhist ? mhist + r * ntiles : NULL);
    }
  }
  free(K);
  free(V);
  free(Vr);
  return 0;
}

/* ------------------------------------ row-sum diagnostic, section 5.5.2 (D1)
 * P: R rows of N nonnegative values (row-major). out: R x 5 doubles per row:
 * sum Q(P), then the zeroing, saturation, downward- and upward-rounding parts
 * of sum(Q(P) - P). rule / q: scale rule as for the quantizers.              */
void orc_rowsum_parts(const double* P, int64_t R, int64_t N, int rule, double q, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; r++) {
    const double* row = P + r * N;
    double sum = 0.0, zero = 0.0, sat = 0.0, down = 0.0, up = 0.0;
    for (int64_t k0 = 0; k0 < N; k0 += ORC_BLOCK) {
      const int n = (int)(N - k0 < ORC_BLOCK ? N - k0 : ORC_BLOCK);
      double v[ORC_BLOCK];
      uint8_t c[ORC_BLOCK];
      for (int i = 0; i < n; i++) v[i] = row[k0 + i];
      const int sbyte = quantize_block(v, n, rule, q, c);
      for (int i = 0; i < n; i++) {
        const double qv = dq(c[i], (uint8_t)sbyte);
        const double d = qv - v[i];
        sum += qv;
        if (v[i] <= 0.0) continue;
        if (qv == 0.0) zero += d;
        else if (ldexp(v[i], 127 - sbyte) > 6.0) sat += d;
        else if (d < 0.0) down += d;
        else if (d > 0.0) up += d;
      }
    }
    out[5 * r + 0] = sum;
    out[5 * r + 1] = zero;
    out[5 * r + 2] = sat;
    out[5 * r + 3] = down;
    out[5 * r + 4] = up;
  }
}

/* ------------------------------------------- unquantized attention, Eq. 1
 * fp64 softmax(Q K^T / sqrt(d)) V on the bf16 inputs (no rotation: an
 * orthogonal rotation leaves QK^T unchanged in exact arithmetic).
 * q, k, v: [BH][N][128] bf16. rows: nrows (bh, token) pairs.                 */
void orc_sdpa(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t BH, int64_t N, int causal,
              const int64_t* rows, int64_t nrows, double* out) {
  (void)BH;
  const double inv_sqrt_d = 1.0 / sqrt((double)ORC_D);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; r++) {
    const int64_t bh = rows[2 * r], i = rows[2 * r + 1];
    const int64_t nk = causal ? i + 1 : N;
    double* s = (double*)malloc(sizeof(double) * nk);
    double qv[ORC_D], acc[ORC_D];
    for (int c = 0; c < ORC_D; c++) {
      qv[c] = bf16_to_f32(q[(bh * N + i) * ORC_D + c]);
      acc[c] = 0.0;
    }
    double mx = -INFINITY;
    for (int64_t j = 0; j < nk; j++) {
      double dot = 0.0;
      for (int c = 0; c < ORC_D; c++) dot += qv[c] * bf16_to_f32(k[(bh * N + j) * ORC_D + c]);
      s[j] = dot * inv_sqrt_d;
      if (s[j] > mx) mx = s[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < nk; j++) {
      double p = exp(s[j] - mx);
      sum += p;
      for (int c = 0; c < ORC_D; c++) acc[c] += p * bf16_to_f32(v[(bh * N + j) * ORC_D + c]);
    }
    for (int c = 0; c < ORC_D; c++) out[r * ORC_D + c] = acc[c] / sum;
    free(s);
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
