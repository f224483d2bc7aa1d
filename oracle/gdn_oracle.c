/*
 * gdn_oracle.c -- plain, sequential fp64 CPU oracle of the Gated DeltaNet (GDN) sublayer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or helper with the CUDA library; it reads bf16 inputs as raw 16-bit patterns
 * and fp32 inputs as floats, and computes everything in double precision, in the order the
 * method defines, one token at a time.
 *
 * What it computes (sources are the pages' titles and sections):
 *   1. causal depthwise conv1d, width W (4), no bias, over the packed [q | k | v] channels,
 *      followed by SiLU and one rounding to bf16 -- pegainfer PR #1152 "Reference golden for
 *      the GDN sublayer", Summary (a four-tap depthwise conv whose only weight is conv1d's) and
 *      "Commands + measured numbers" (the conv leg is a bf16 tensor compared bit-exact);
 *      GLM-5.3-Flash kernel TDD ledger, slice I3 (the decode step equals the full width-4
 *      causal convolution).
 *   2. head expansion q/k by repeat_interleave (V head h reads K head h / (Hv/Hk)) and L2
 *      normalisation x / sqrt(sum x^2 + eps) -- PR #1152 Summary (V/K ratio 3,
 *      repeat_interleave) and its Code review (prepare: head expand + L2 norm);
 *      GLM-5.3-Flash ledger slice I2a (independent x/sqrt(sum(x^2)+eps), not max(norm, eps),
 *      not an RMS norm).
 *   3. the gated delta rule with an fp32 [value, key] state carried across chunks, calls and
 *      sequences:  S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *      o_t = q_scale * S_t q_t  -- PR #1152 Code review (f32 recurrent state, cross-chunk
 *      carry); GLM-5.3-Flash ledger slice I2 (an fp32 state indexed [value, key], its own q scale).
 *      It is evaluated as its expanded form: S <- exp(g) S;  e = beta (v - S k);  S <- S + e k^T.
 *   4. gated RMSNorm with a sigmoid output gate: out = o * (mean(o^2) + eps)^-1/2 * w * sigmoid(z)
 *      -- PR #1152 Summary (output_gate_type "sigmoid", not silu) and Code review item 6
 *      (rms_norm_eps == 1e-6).
 *   5. the one-token decode step: conv step on a (W-1)-deep shift register of raw inputs,
 *      then steps 2-4 for one token -- Qwen3.8 kernel architecture and TDD ledger, "Current
 *      dense-27B kernel map" (scalar GDN recurrence and fused output gate).
 *   6. the same decode step with the recurrent state stored as IEEE binary16: widened on load,
 *      the step in double, rounded once (ties to even) on store -- the same ledger, the FP16
 *      h-state twins of the decode kernels.
 *   7. the gates g and beta from the a / b projections, A_log and dt_bias (parity unpinned: the
 *      pages give no formula; the published Gated DeltaNet / Mamba-2 gate is taken).
 *   8. the KDA decode step: the same with a per-channel (key-dimension) decay, clamped and
 *      exponentiated -- GLM-5.3-Flash kernel TDD ledger, slices I2, I2a, I3.
 *   9. the KDA recurrence over packed sequences (the prefill's sequential form): step 3 with the
 *      decay of item 8, token by token -- the same ledger, slice I4 (the chunk path must match
 *      the sequential state and output).
 *
 * Mutations (negative controls) can be planted here, on the CPU, through the `mutation`
 * bit set; 0 is the method.  See ORACLE_MUT_* below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_MUT_SILU_GATE 0x001 /* gate by z*sigmoid(z) instead of sigmoid(z)            */
#define ORACLE_MUT_NO_CONV 0x002   /* skip the conv leg: q|k|v = raw input                  */
#define ORACLE_MUT_DROP_CARRY 0x004 /* restart from the initial state at every 64th token */
#define ORACLE_MUT_TRANSPOSE 0x008 /* read/write the state as [key, value]                  */
#define ORACLE_MUT_TILED_HEADS 0x010 /* V head h reads K head h % Hk                        */
#define ORACLE_MUT_CONV_SHIFT 0x020 /* conv window shifted one position into the past       */
#define ORACLE_MUT_DECAY_SIGN 0x040 /* decay by exp(-g)                                     */
#define ORACLE_MUT_NO_BETA 0x080    /* beta forced to 1                                     */
#define ORACLE_MUT_NO_QNORM 0x100   /* q is not L2-normalised                               */

/* ---------------------------------------------------------------- bf16 <-> double */

static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (1 sign, 8 exponent, 7 stored mantissa bits), ties to
 * even, directly from the exact value (no intermediate rounding to float). */
uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double ax = fabs(x);
  if (ax == 0.0) return sign;
  if (isinf(ax)) return sign | 0x7F80;
  int e;
  (void)frexp(ax, &e);           /* ax = m * 2^e, 0.5 <= m < 1: leading bit weighs 2^(e-1) */
  int qexp = e - 8;              /* 8 significant bits -> quantum 2^(e-8)                  */
  if (qexp < -133) qexp = -133;  /* subnormal bf16 quantum is 2^-133                       */
  double r = nearbyint(ldexp(ax, -qexp)); /* round to integer, ties to even                 */
  double y = ldexp(r, qexp);
  if (y > 3.3895313892515355e38) return sign | 0x7F80; /* above the largest finite bf16   */
  float f = (float)y;            /* exact: y has at most 8 significant bits                */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ---------------------------------------------------------------- 1. conv1d + SiLU (prefill) */

/*
 * x:          [T, C] bf16 raw conv input (packed q|k|v channels, token-major)
 * w:          [C, W] bf16; w[c, W-1] multiplies the current token, w[c, 0] the oldest
 * cu_seqlens: [N+1] token offsets of the packed sequences
 * state_in:   [N, C, W-1] bf16 raw inputs preceding each sequence, oldest first, or NULL (zeros)
 * y:          [T, C] bf16 = round_bf16(silu(sum_i w[c,i] x[t-(W-1)+i, c]))
 * y_exact:    [T, C] double, the same before rounding, or NULL
 * state_out:  [N, C, W-1] bf16, the last W-1 raw inputs of each sequence (history shifted in)
 */
int oracle_conv1d_prefill(int C, int W, int T, const uint16_t* x, const uint16_t* w,
                          const int32_t* cu_seqlens, int N, const uint16_t* state_in,
                          uint16_t* y, double* y_exact, uint16_t* state_out, int mutation) {
  if (C <= 0 || W < 1 || T < 0 || N < 0) return 1;
  if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return 2;
  for (int n = 0; n < N; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
  const int H = W - 1;
  for (int n = 0; n < N; ++n) {
    const int s = cu_seqlens[n], L = cu_seqlens[n + 1] - s;
    for (int c = 0; c < C; ++c) {
      /* value of the raw input at position p relative to the sequence start (p may be < 0) */
#define RAW(p) ((p) >= 0 ? bf16_to_double(x[(size_t)(s + (p)) * C + c])                     \
                         : ((p) >= -H && state_in                                           \
                                ? bf16_to_double(state_in[((size_t)n * C + c) * H + H + (p)]) \
                                : 0.0))
      for (int t = 0; t < L; ++t) {
        double a;
        if (mutation & ORACLE_MUT_NO_CONV) {
          a = RAW(t);
        } else {
          double acc = 0.0;
          for (int i = 0; i < W; ++i) {
            int p = t - H + i;
            if (mutation & ORACLE_MUT_CONV_SHIFT) p -= 1;
            acc += bf16_to_double(w[(size_t)c * W + i]) * RAW(p);
          }
          a = acc * sigmoid(acc); /* SiLU */
        }
        if (y_exact) y_exact[(size_t)(s + t) * C + c] = a;
        if (y) y[(size_t)(s + t) * C + c] = oracle_round_bf16(a);
      }
      if (state_out && H > 0) {
        /* read every slot before writing so that state_out may alias state_in */
        double slot[16];
        for (int j = 0; j < H && j < 16; ++j) slot[j] = RAW(L - H + j);
        for (int j = 0; j < H && j < 16; ++j)
          state_out[((size_t)n * C + c) * H + j] = oracle_round_bf16(slot[j]);
      }
#undef RAW
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- 2+3. the recurrence */

typedef struct {
  int hk, hv, dk, dv;
  const uint16_t* qkv;   /* [T, 2*hk*dk + hv*dv] bf16 */
  const float* g;        /* [T, hv], or NULL when gk is given */
  const float* gk;       /* [T, hv, dk] per-key-channel log decay (KDA), or NULL */
  double g_min;          /* clamp of gk: exp(max(gk, g_min)) */
  const float* beta;     /* [T, hv] */
  const int32_t* cu;     /* [N+1] */
  int N;
  double q_scale, l2_eps;
  const double* state_in; /* [N, hv, dv, dk] or NULL */
  double* o;              /* [T, hv, dv] */
  double* state_out;      /* [N, hv, dv, dk] or NULL */
  const int32_t* heads;   /* subset of V heads to compute, or NULL for all */
  int nheads;
  int mutation;
  long next;              /* work counter */
  pthread_mutex_t lock;
} rec_job;

static void rec_chain(rec_job* J, int n, int h) {
  const int hk = J->hk, hv = J->hv, dk = J->dk, dv = J->dv;
  const int C = 2 * hk * dk + hv * dv;
  const int ratio = hv / hk;
  const int j = (J->mutation & ORACLE_MUT_TILED_HEADS) ? (h % hk) : (h / ratio);
  const size_t sdim = (size_t)dv * dk;
  double* S = (double*)malloc(sizeof(double) * sdim);
  double* S0 = (double*)malloc(sizeof(double) * sdim);
  double* qn = (double*)malloc(sizeof(double) * dk);
  double* kn = (double*)malloc(sizeof(double) * dk);
  double* e = (double*)malloc(sizeof(double) * dv);
  /* S[r*dk + i]: row r = value index, column i = key index ([value, key] layout) */
  for (int r = 0; r < dv; ++r)
    for (int i = 0; i < dk; ++i) {
      double v0 = 0.0;
      if (J->state_in) {
        const double* si = J->state_in + ((size_t)n * hv + h) * sdim;
        v0 = (J->mutation & ORACLE_MUT_TRANSPOSE) ? si[(size_t)i * dv + r] : si[(size_t)r * dk + i];
      }
      S0[(size_t)r * dk + i] = v0;
      S[(size_t)r * dk + i] = v0;
    }
  const int s = J->cu[n], L = J->cu[n + 1] - s;
  for (int tt = 0; tt < L; ++tt) {
    const size_t t = (size_t)(s + tt);
    if ((J->mutation & ORACLE_MUT_DROP_CARRY) && tt > 0 && tt % 64 == 0)
      memcpy(S, S0, sizeof(double) * sdim);
    const uint16_t* row = J->qkv + t * C;
    /* L2 normalisation of q and k of K head j (x / sqrt(sum x^2 + eps)) */
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < dk; ++i) {
      double qv = bf16_to_double(row[j * dk + i]);
      double kv = bf16_to_double(row[hk * dk + j * dk + i]);
      qn[i] = qv;
      kn[i] = kv;
      sq += qv * qv;
      sk += kv * kv;
    }
    const double iq = (J->mutation & ORACLE_MUT_NO_QNORM) ? 1.0 : 1.0 / sqrt(sq + J->l2_eps);
    const double ik = 1.0 / sqrt(sk + J->l2_eps);
    for (int i = 0; i < dk; ++i) {
      qn[i] *= iq;
      kn[i] *= ik;
    }
    const double b = (J->mutation & ORACLE_MUT_NO_BETA) ? 1.0 : (double)J->beta[t * hv + h];
    const uint16_t* vrow = row + 2 * hk * dk + (size_t)h * dv;
    /* decay, then the delta correction against the decayed state */
    if (J->gk) {
      /* KDA: key column i of the [value, key] state decays by exp(max(g_i, g_min)) */
      const float* gv = J->gk + (t * hv + h) * dk;
      for (int i = 0; i < dk; ++i) {
        const double gi = (double)gv[i] > J->g_min ? (double)gv[i] : J->g_min;
        const double ai = exp((J->mutation & ORACLE_MUT_DECAY_SIGN) ? -gi : gi);
        for (int r = 0; r < dv; ++r) S[(size_t)r * dk + i] *= ai;
      }
    } else {
      const double gt = (double)J->g[t * hv + h];
      const double alpha = exp((J->mutation & ORACLE_MUT_DECAY_SIGN) ? -gt : gt);
      for (size_t x = 0; x < sdim; ++x) S[x] *= alpha;
    }
    for (int r = 0; r < dv; ++r) {
      double u = 0.0;
      for (int i = 0; i < dk; ++i) u += S[(size_t)r * dk + i] * kn[i];
      e[r] = b * (bf16_to_double(vrow[r]) - u);
    }
    for (int r = 0; r < dv; ++r)
      for (int i = 0; i < dk; ++i) S[(size_t)r * dk + i] += e[r] * kn[i];
    /* o_t = q_scale * S_t q_t */
    double* orow = J->o + (t * hv + h) * dv;
    for (int r = 0; r < dv; ++r) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * qn[i];
      orow[r] = J->q_scale * acc;
    }
  }
  if (J->state_out) {
    double* so = J->state_out + ((size_t)n * hv + h) * sdim;
    for (int r = 0; r < dv; ++r)
      for (int i = 0; i < dk; ++i) {
        if (J->mutation & ORACLE_MUT_TRANSPOSE)
          so[(size_t)i * dv + r] = S[(size_t)r * dk + i];
        else
          so[(size_t)r * dk + i] = S[(size_t)r * dk + i];
      }
  }
  free(S); free(S0); free(qn); free(kn); free(e);
}

static void* rec_worker(void* arg) {
  rec_job* J = (rec_job*)arg;
  const long nh = J->heads ? J->nheads : J->hv;
  const long total = (long)J->N * nh;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    long w = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (w >= total) break;
    int n = (int)(w / nh);
    int h = J->heads ? J->heads[w % nh] : (int)(w % nh);
    rec_chain(J, n, h);
  }
  return NULL;
}

int oracle_num_threads(void) {
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

/* runs every chain of the job on nthreads workers (<= 0: all online cores) */
static void run_chains(rec_job* J, int nthreads) {
  J->next = 0;
  pthread_mutex_init(&J->lock, NULL);
  if (nthreads <= 0) nthreads = oracle_num_threads();
  const long work = (long)J->N * (J->heads ? J->nheads : J->hv);
  if (nthreads > work) nthreads = work > 0 ? (int)work : 1;
  if (nthreads <= 1) {
    rec_worker(J);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, rec_worker, J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&J->lock);
}

/*
 * The gated delta rule over packed variable-length sequences (one chain per (sequence, V head)).
 * qkv:      [T, 2*hk*dk + hv*dv] bf16 conv output: q heads, then k heads, then v heads
 * g, beta:  [T, hv] fp32 (log decay and write strength)
 * state_in: [N, hv, dv, dk] double initial states ([value, key]) or NULL for zeros
 * o:        [T, hv, dv] double;  state_out: [N, hv, dv, dk] double or NULL
 * heads:    optional list of V heads to compute (the other heads of o/state_out are untouched)
 * nthreads: worker threads over the independent chains (<= 0: all online cores)
 */
int oracle_gdn_recurrence(int hk, int hv, int dk, int dv, int T, const uint16_t* qkv,
                          const float* g, const float* beta, const int32_t* cu_seqlens, int N,
                          double q_scale, double l2_eps, const double* state_in, double* o,
                          double* state_out, const int32_t* heads, int nheads, int nthreads,
                          int mutation) {
  if (hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0 || hv % hk != 0 || N < 0) return 1;
  if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return 2;
  for (int n = 0; n < N; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
  rec_job J;
  J.hk = hk; J.hv = hv; J.dk = dk; J.dv = dv;
  J.qkv = qkv; J.g = g; J.gk = NULL; J.g_min = 0.0; J.beta = beta; J.cu = cu_seqlens; J.N = N;
  J.q_scale = q_scale; J.l2_eps = l2_eps;
  J.state_in = state_in; J.o = o; J.state_out = state_out;
  J.heads = heads; J.nheads = nheads; J.mutation = mutation;
  run_chains(&J, nthreads);
  return 0;
}

/*
 * The KDA recurrence over packed variable-length sequences: as oracle_gdn_recurrence, with
 * g: [T, hv, dk] fp32, a log decay per key channel, applied as exp(max(g, g_min)) to the key
 * columns of the [value, key] state (g_min = -inf: no clamp).
 */
int oracle_kda_recurrence(int hk, int hv, int dk, int dv, int T, const uint16_t* qkv,
                          const float* g, double g_min, const float* beta,
                          const int32_t* cu_seqlens, int N, double q_scale, double l2_eps,
                          const double* state_in, double* o, double* state_out,
                          const int32_t* heads, int nheads, int nthreads, int mutation) {
  if (hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0 || hv % hk != 0 || N < 0) return 1;
  if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return 2;
  for (int n = 0; n < N; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
  rec_job J;
  J.hk = hk; J.hv = hv; J.dk = dk; J.dv = dv;
  J.qkv = qkv; J.g = NULL; J.gk = g; J.g_min = g_min; J.beta = beta; J.cu = cu_seqlens; J.N = N;
  J.q_scale = q_scale; J.l2_eps = l2_eps;
  J.state_in = state_in; J.o = o; J.state_out = state_out;
  J.heads = heads; J.nheads = nheads; J.mutation = mutation;
  run_chains(&J, nthreads);
  return 0;
}

/* ---------------------------------------------------------------- 4. gated RMSNorm */

/*
 * o:   [rows, dv] double (rows = tokens * V heads), z: [rows, dv] bf16, w: [dv] bf16
 * out: [rows, dv] double = o * (mean_d o^2 + eps)^(-1/2) * w * sigmoid(z)
 */
int oracle_gated_rmsnorm(long rows, int dv, const double* o, const uint16_t* z,
                         const uint16_t* w, double eps, double* out, int mutation) {
  for (long r = 0; r < rows; ++r) {
    const double* orow = o + (size_t)r * dv;
    double ss = 0.0;
    for (int d = 0; d < dv; ++d) ss += orow[d] * orow[d];
    const double inv = 1.0 / sqrt(ss / dv + eps);
    for (int d = 0; d < dv; ++d) {
      const double zz = bf16_to_double(z[(size_t)r * dv + d]);
      const double gate = (mutation & ORACLE_MUT_SILU_GATE) ? zz * sigmoid(zz) : sigmoid(zz);
      out[(size_t)r * dv + d] = orow[d] * inv * bf16_to_double(w[d]) * gate;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- 5. decode step */

/*
 * One token for each of B independent sequences.
 * x:          [B, C] bf16 raw conv input of this step
 * conv_state: [B, C, W-1] bf16 in/out shift register of the previous W-1 raw inputs, oldest first
 * state:      [B, hv, dv, dk] double in/out recurrent state
 * g, beta:    [B, hv] fp32;  z: [B, hv, dv] bf16;  norm_w: [dv] bf16
 * out:        [B, hv, dv] double gated output;  o_raw: [B, hv, dv] double or NULL (pre-norm)
 */
/* The conv step of one token for B sequences: window = [state[0..H-1], x];
 * y = sum_i w[c,i] window[i]; a = bf16(y * sigmoid(y)); state <- window[1..H]. */
static void conv_decode_step(int C, int W, int B, const uint16_t* x, const uint16_t* conv_w,
                             uint16_t* conv_state, uint16_t* a, int mutation) {
  const int H = W - 1;
  for (int b = 0; b < B; ++b) {
    for (int c = 0; c < C; ++c) {
      double win[17];
      uint16_t* st = conv_state + ((size_t)b * C + c) * H;
      for (int i = 0; i < H; ++i) win[i] = bf16_to_double(st[i]);
      win[H] = bf16_to_double(x[(size_t)b * C + c]);
      double acc = 0.0;
      if (mutation & ORACLE_MUT_CONV_SHIFT) {
        for (int i = 1; i < W; ++i) acc += bf16_to_double(conv_w[(size_t)c * W + i]) * win[i - 1];
      } else {
        for (int i = 0; i < W; ++i) acc += bf16_to_double(conv_w[(size_t)c * W + i]) * win[i];
      }
      const double act = (mutation & ORACLE_MUT_NO_CONV) ? win[H] : acc * sigmoid(acc);
      a[(size_t)b * C + c] = oracle_round_bf16(act);
      for (int i = 0; i < H; ++i) st[i] = oracle_round_bf16(win[i + 1]);
    }
  }
}

int oracle_decode_step(int hk, int hv, int dk, int dv, int W, int B, const uint16_t* x,
                       const uint16_t* conv_w, uint16_t* conv_state, const float* g,
                       const float* beta, double* state, const uint16_t* z,
                       const uint16_t* norm_w, double q_scale, double l2_eps, double rms_eps,
                       double* out, double* o_raw, int nthreads, int mutation) {
  const int C = 2 * hk * dk + hv * dv;
  uint16_t* a = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)B * C);
  double* o = o_raw ? o_raw : (double*)malloc(sizeof(double) * (size_t)B * hv * dv);
  int32_t* cu = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B + 1));
  conv_decode_step(C, W, B, x, conv_w, conv_state, a, mutation);
  for (int b = 0; b <= B; ++b) cu[b] = b;
  int rc = oracle_gdn_recurrence(hk, hv, dk, dv, B, a, g, beta, cu, B, q_scale, l2_eps, state, o,
                                 state, NULL, 0, nthreads, mutation & ~ORACLE_MUT_DROP_CARRY);
  if (rc == 0) rc = oracle_gated_rmsnorm((long)B * hv, dv, o, z, norm_w, rms_eps, out, mutation);
  free(a);
  free(cu);
  if (!o_raw) free(o);
  return rc;
}

/* ---------------------------------------------------------------- 6. decode with an fp16 state */

/* IEEE 754 binary16 (1 sign, 5 exponent bits with bias 15, 10 stored mantissa bits) -> double.
 * Exponent field 0 holds zero and the subnormals (mantissa * 2^-24); field 31 holds the
 * infinities and NaNs. */
double oracle_f16_to_double(uint16_t h) {
  const double sign = (h & 0x8000) ? -1.0 : 1.0;
  const int ex = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  if (ex == 0x1F) return man ? NAN : sign * INFINITY;
  if (ex == 0) return sign * ldexp((double)man, -24);
  return sign * ldexp((double)(0x400 | man), ex - 25);
}

/* Round a double to the nearest binary16, ties to even, directly from the exact value.  Values
 * whose rounded magnitude exceeds the largest finite binary16 (65504) become infinities. */
uint16_t oracle_round_f16(double x) {
  if (isnan(x)) return 0x7E00;
  const uint16_t sign = signbit(x) ? 0x8000 : 0;
  const double ax = fabs(x);
  if (ax == 0.0) return sign;
  if (isinf(ax)) return sign | 0x7C00;
  int e;
  (void)frexp(ax, &e);          /* ax = m * 2^e, 0.5 <= m < 1: leading bit weighs 2^(e-1) */
  int qexp = e - 11;            /* 11 significant bits -> quantum 2^(e-11)                */
  if (qexp < -24) qexp = -24;   /* subnormal binary16 quantum is 2^-24                    */
  const double r = nearbyint(ldexp(ax, -qexp)); /* round to integer, ties to even          */
  const double y = ldexp(r, qexp);
  if (y > 65504.0) return sign | 0x7C00;
  if (y < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(y, 24); /* subnormal (or zero)   */
  int ey;
  const double my = frexp(y, &ey);                   /* y = my * 2^ey, my in [0.5, 1)        */
  const int field = ey - 1 + 15;                     /* biased exponent of the leading bit   */
  const int mant = (int)ldexp(my, 11) - 0x400;       /* the 10 bits below the leading one    */
  return sign | (uint16_t)(field << 10) | (uint16_t)mant;
}

/*
 * oracle_decode_step with the recurrent state held as binary16 in memory: every element is
 * widened to double, the step runs exactly as oracle_decode_step (the output from the new state
 * as computed, before any rounding), and the new state is rounded once to binary16 when it is
 * stored.  Qwen3.8 kernel architecture and TDD ledger, the FP16 h-state twins of the decode and
 * WY kernels (the FP32 kernels' arithmetic, with the state stored in half precision and rounded
 * whenever a token's state is stored).
 * state_h: [B, hv, dv, dk] binary16 bit patterns, in/out.  Other arguments as oracle_decode_step.
 */
int oracle_decode_step_h16(int hk, int hv, int dk, int dv, int W, int B, const uint16_t* x,
                           const uint16_t* conv_w, uint16_t* conv_state, const float* g,
                           const float* beta, uint16_t* state_h, const uint16_t* z,
                           const uint16_t* norm_w, double q_scale, double l2_eps, double rms_eps,
                           double* out, double* o_raw, int nthreads, int mutation) {
  const size_t n = (size_t)B * hv * dv * dk;
  double* st = (double*)malloc(sizeof(double) * (n ? n : 1));
  if (!st) return -1;
  for (size_t i = 0; i < n; ++i) st[i] = oracle_f16_to_double(state_h[i]);
  const int rc = oracle_decode_step(hk, hv, dk, dv, W, B, x, conv_w, conv_state, g, beta, st, z,
                                    norm_w, q_scale, l2_eps, rms_eps, out, o_raw, nthreads,
                                    mutation);
  if (rc == 0)
    for (size_t i = 0; i < n; ++i) state_h[i] = oracle_round_f16(st[i]);
  free(st);
  return rc;
}

/* ---------------------------------------------------------------- 7. gate derivation */

/*
 * The per-token gates from their projections (PARITY UNPINNED: the pages name the inputs -- the
 * a / b projections, A_log and dt_bias, Qwen3.8 kernel architecture and TDD ledger, the kernel
 * map's GDN gate transforms; PR #1152 Summary -- but give no formula).  The reading taken is the
 * gate of the published Gated DeltaNet / Mamba-2 layers:
 *   g[t,h]    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h]),   softplus(x) = log(1 + e^x)
 *   beta[t,h] = sigmoid(b[t,h]) = 1 / (1 + e^-b)
 * a, b: [rows, hv] bf16;  A_log, dt_bias: [hv] fp32;  g, beta: [rows, hv] double.
 */
int oracle_gates(long rows, int hv, const uint16_t* a, const uint16_t* b, const float* A_log,
                 const float* dt_bias, double* g, double* beta) {
  for (long t = 0; t < rows; ++t)
    for (int h = 0; h < hv; ++h) {
      const size_t i = (size_t)t * hv + h;
      const double x = bf16_to_double(a[i]) + (double)dt_bias[h];
      const double sp = x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); /* log(1 + e^x), no overflow */
      g[i] = -exp((double)A_log[h]) * sp;
      beta[i] = sigmoid(bf16_to_double(b[i]));
    }
  return 0;
}

/* ---------------------------------------------------------------- 8. KDA decode step */

/*
 * One token of the KDA (Kimi delta attention) layer for each of B sequences: the gated delta
 * rule with a per-channel (key-dimension) decay -- GLM-5.3-Flash kernel TDD ledger, slices I2
 * (an fp32 state indexed [value, key], the decay clamped then exponentiated, its own q scale), I2a
 * (q/k normalised x / sqrt(sum x^2 + eps)) and I3 (the width-4 conv step).  Per V head h,
 * with q, k of K head h / (hv/hk) after the conv step and the L2 norms:
 *   alpha_i = exp(max(g[b,h,i], g_min))        (g_min = -inf: no clamp)
 *   S[r][i] <- alpha_i S[r][i];   e_r = beta (v_r - sum_i S[r][i] k_i);   S[r][i] += e_r k_i
 *   o_r = q_scale sum_i S[r][i] q_i;   out = gated RMSNorm(o, z) as for the GDN layer.
 * g: [B, hv, dk] fp32 (per-channel log decay); beta: [B, hv]; state [B, hv, dv, dk] double
 * in/out; other arguments as oracle_decode_step.
 */
int oracle_kda_decode_step(int hk, int hv, int dk, int dv, int W, int B, const uint16_t* x,
                           const uint16_t* conv_w, uint16_t* conv_state, const float* g,
                           double g_min, const float* beta, double* state, const uint16_t* z,
                           const uint16_t* norm_w, double q_scale, double l2_eps, double rms_eps,
                           double* out, double* o_raw, int mutation) {
  if (hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0 || hv % hk != 0 || B < 0) return 1;
  const int C = 2 * hk * dk + hv * dv;
  const int ratio = hv / hk;
  uint16_t* a = (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)B * C + 1));
  double* o = o_raw ? o_raw : (double*)malloc(sizeof(double) * ((size_t)B * hv * dv + 1));
  double* qn = (double*)malloc(sizeof(double) * dk);
  double* kn = (double*)malloc(sizeof(double) * dk);
  double* e = (double*)malloc(sizeof(double) * dv);
  conv_decode_step(C, W, B, x, conv_w, conv_state, a, mutation);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < hv; ++h) {
      const int j = h / ratio;
      const uint16_t* row = a + (size_t)b * C;
      double sq = 0.0, sk = 0.0;
      for (int i = 0; i < dk; ++i) {
        qn[i] = bf16_to_double(row[j * dk + i]);
        kn[i] = bf16_to_double(row[hk * dk + j * dk + i]);
        sq += qn[i] * qn[i];
        sk += kn[i] * kn[i];
      }
      const double iq = (mutation & ORACLE_MUT_NO_QNORM) ? 1.0 : 1.0 / sqrt(sq + l2_eps);
      const double ik = 1.0 / sqrt(sk + l2_eps);
      for (int i = 0; i < dk; ++i) {
        qn[i] *= iq;
        kn[i] *= ik;
      }
      double* S = state + ((size_t)b * hv + h) * dv * dk;
      const float* gv = g + ((size_t)b * hv + h) * dk;
      const double bt = (mutation & ORACLE_MUT_NO_BETA) ? 1.0 : (double)beta[(size_t)b * hv + h];
      const uint16_t* vrow = row + 2 * hk * dk + (size_t)h * dv;
      /* element (r, i) of the [value, key] state; the transposed mutation reads it as [key, value] */
#define SEL(r, i) (*((mutation & ORACLE_MUT_TRANSPOSE) ? &S[(size_t)(i) * dv + (r)] : &S[(size_t)(r) * dk + (i)]))
      for (int r = 0; r < dv; ++r)
        for (int i = 0; i < dk; ++i) {
          const double gi = (double)gv[i] > g_min ? (double)gv[i] : g_min;
          SEL(r, i) *= exp((mutation & ORACLE_MUT_DECAY_SIGN) ? -gi : gi);
        }
      for (int r = 0; r < dv; ++r) {
        double u = 0.0;
        for (int i = 0; i < dk; ++i) u += SEL(r, i) * kn[i];
        e[r] = bt * (bf16_to_double(vrow[r]) - u);
      }
      for (int r = 0; r < dv; ++r)
        for (int i = 0; i < dk; ++i) SEL(r, i) += e[r] * kn[i];
      double* orow = o + ((size_t)b * hv + h) * dv;
      for (int r = 0; r < dv; ++r) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += SEL(r, i) * qn[i];
        orow[r] = q_scale * acc;
      }
#undef SEL
    }
  const int rc = oracle_gated_rmsnorm((long)B * hv, dv, o, z, norm_w, rms_eps, out, mutation);
  free(a);
  free(qn);
  free(kn);
  free(e);
  if (!o_raw) free(o);
  return rc;
}
