/*
 * oracle.c -- plain CPU checker for the sharded mixed-precision AdamW step.
 * TEST INFRASTRUCTURE ONLY (see oracle.h). Build: -O2 -ffp-contract=off
 * -fno-fast-math, so each C statement below is one IEEE operation rounded to
 * nearest-even and no multiply-add is fused.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORC_NORM_CHUNK (1 << 20)

static int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

/* ================================================================= plan ==== */

int orc_plan_make(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                  int64_t bucket_elems, orc_plan* out, int64_t* offsets,
                  orc_segment* segs, int32_t seg_cap) {
  if (!out || n_tensors < 0 || n_ranks < 1 || bucket_elems < 0) return -1;
  if (n_tensors > 0 && !numels) return -1;
  memset(out, 0, sizeof(*out));
  /* flatten: tensor k starts where the previous tensors end */
  int64_t psi = 0;
  for (int32_t k = 0; k < n_tensors; ++k) {
    if (numels[k] < 0) return -1;
    if (offsets) offsets[k] = psi;
    psi += numels[k];
  }
  /* pad to a multiple of N and give rank i the slice [i*S, (i+1)*S) */
  int64_t pad = (n_ranks - psi % n_ranks) % n_ranks;
  int64_t psi_pad = psi + pad;
  int64_t shard = psi_pad / n_ranks;
  out->psi = psi;
  out->pad = pad;
  out->psi_pad = psi_pad;
  out->shard = shard;
  out->bucket_elems = bucket_elems;
  out->n_ranks = n_ranks;

  /* buckets of B elements over the padded flat buffer (B = 0: one bucket) */
  int64_t nb = 0;
  if (psi_pad > 0) nb = bucket_elems == 0 ? 1 : (psi_pad + bucket_elems - 1) / bucket_elems;
  out->n_buckets = (int32_t)nb;

  /* segments: each bucket cut at the owners' slice boundaries */
  int32_t ns = 0;
  for (int64_t k = 0; k < nb; ++k) {
    int64_t blo = bucket_elems == 0 ? 0 : k * bucket_elems;
    int64_t bhi = bucket_elems == 0 ? psi_pad : imin64((k + 1) * bucket_elems, psi_pad);
    for (int32_t i = 0; i < n_ranks; ++i) {
      int64_t lo = imax64(blo, (int64_t)i * shard);
      int64_t hi = imin64(bhi, (int64_t)(i + 1) * shard);
      if (lo >= hi) continue;
      if (segs && ns < seg_cap) {
        segs[ns].lo = lo;
        segs[ns].hi = hi;
        segs[ns].rank = i;
        segs[ns].bucket = (int32_t)k;
      }
      ++ns;
    }
  }
  out->n_segments = ns;

  double b[4];
  orc_bills((double)psi, n_ranks, b);
  out->bill_ddp = b[0];
  out->bill_z1 = b[1];
  out->bill_z2 = b[2];
  out->bill_z3 = b[3];
  out->ring_bytes_per_rank = orc_ring_bytes(2.0 * (double)psi, n_ranks);
  out->ring_hops = 2.0 * (double)(n_ranks - 1);
  /* [SR] "FSDP: the same idea, layer-native" and [SB] "What does each stage
   * cost on the wire?": 2 psi for DDP and stages 1-2, 3 psi for stage 3 */
  out->comm_ddp = 2.0 * (double)psi;
  out->comm_z1 = 2.0 * (double)psi;
  out->comm_z2 = 2.0 * (double)psi;
  out->comm_z3 = 3.0 * (double)psi;
  if (segs && ns > seg_cap) return -2;
  return 0;
}

void orc_bills(double psi, int32_t n_ranks, double out[4]) {
  const double K = 12.0; /* fp32 master + m + v, 4 bytes each */
  const double N = (double)n_ranks;
  out[0] = (2.0 + 2.0 + K) * psi;             /* baseline DP */
  out[1] = (2.0 + 2.0) * psi + K * psi / N;   /* P_os */
  out[2] = 2.0 * psi + (2.0 + K) * psi / N;   /* P_os+g */
  out[3] = (2.0 + 2.0 + K) * psi / N;         /* P_os+g+p */
}

double orc_ring_bytes(double m_bytes, int32_t d) {
  return 2.0 * (double)(d - 1) * m_bytes / (double)d;
}

/* ================================================================ casts ==== */

/* Encoder for a binary format with `ebits` exponent bits, `mbits` fraction
 * bits and bias 2^(ebits-1)-1, from the IEEE 754 definition: write the fp32
 * input as sig * 2^q with an integer significand, pick the target exponent
 * Et = max(floor(log2 |x|), emin), keep the multiple n of the quantum
 * 2^(Et - mbits) nearest to |x| (ties to the even multiple), carry into the
 * next binade when n reaches 2^(mbits+1), overflow to infinity above the
 * largest exponent, and encode n as a subnormal (n < 2^mbits) or normal. */
static uint16_t encode_small_float(float x, int ebits, int mbits) {
  uint32_t u;
  memcpy(&u, &x, 4);
  const uint32_t sign = (u >> 31) << (ebits + mbits);
  const uint32_t exp_all = ((1u << ebits) - 1u) << mbits;
  const uint32_t e32 = (u >> 23) & 0xFFu;
  const uint32_t f32 = u & 0x7FFFFFu;
  if (e32 == 0xFFu) /* infinity, or NaN made quiet */
    return (uint16_t)(f32 ? (sign | exp_all | (1u << (mbits - 1))) : (sign | exp_all));
  if (e32 == 0 && f32 == 0) return (uint16_t)sign;
  const int bias = (1 << (ebits - 1)) - 1;
  const int emin = 1 - bias, emax = bias;
  /* |x| = sig * 2^q */
  uint32_t sig = e32 ? (f32 | 0x800000u) : f32;
  int q = e32 ? (int)e32 - 127 - 23 : -126 - 23;
  int nb = 0;
  for (uint32_t t = sig; t; t >>= 1) ++nb; /* bit length of sig */
  int Et = q + nb - 1;
  if (Et < emin) Et = emin;
  int shift = (Et - mbits) - q; /* low bits of sig below the quantum */
  uint32_t n;
  if (shift <= 0) {
    n = sig << (-shift);
  } else if (shift >= 25) {
    n = 0; /* below half a quantum (sig < 2^24) */
  } else {
    n = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (n & 1u))) n += 1;
  }
  if (n == (2u << mbits)) { /* rounded up into the next binade */
    n >>= 1;
    Et += 1;
  }
  if (Et > emax) return (uint16_t)(sign | exp_all);
  if (n < (1u << mbits)) return (uint16_t)(sign | n); /* subnormal or zero */
  return (uint16_t)(sign | ((uint32_t)(Et + bias) << mbits) | (n - (1u << mbits)));
}

/* Decoder: subnormals are frac * 2^(emin - mbits) (exact in fp32), normals
 * get the fp32 exponent field e - bias + 127 and the fraction shifted into
 * the top of fp32's 23 fraction bits. */
static float decode_small_float(uint16_t h, int ebits, int mbits) {
  const int bias = (1 << (ebits - 1)) - 1;
  const uint32_t sign = ((uint32_t)h >> (ebits + mbits)) & 1u;
  const uint32_t ef = ((uint32_t)h >> mbits) & ((1u << ebits) - 1u);
  const uint32_t fr = (uint32_t)h & ((1u << mbits) - 1u);
  uint32_t bits;
  if (ef == (1u << ebits) - 1u) {
    bits = 0x7F800000u | (fr << (23 - mbits));
  } else if (ef == 0) {
    float mag = (float)fr * ldexpf(1.0f, 1 - bias - mbits);
    memcpy(&bits, &mag, 4);
  } else {
    bits = ((ef - (uint32_t)bias + 127u) << 23) | (fr << (23 - mbits));
  }
  bits |= sign << 31;
  float out;
  memcpy(&out, &bits, 4);
  return out;
}

uint16_t orc_f32_to_f16(float x) { return encode_small_float(x, 5, 10); }
float orc_f16_to_f32(uint16_t h) { return decode_small_float(h, 5, 10); }
uint16_t orc_f32_to_bf16(float x) { return encode_small_float(x, 8, 7); }
float orc_bf16_to_f32(uint16_t h) { return decode_small_float(h, 8, 7); }

static uint16_t cast16(float x, int32_t is_bf16) {
  return is_bf16 ? orc_f32_to_bf16(x) : orc_f32_to_f16(x);
}
static float widen16(uint16_t h, int32_t is_bf16) {
  return is_bf16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

void orc_cast_array(const float* in, uint16_t* out, int64_t n, int32_t is_bf16) {
  for (int64_t k = 0; k < n; ++k) out[k] = cast16(in[k], is_bf16);
}
void orc_widen_array(const uint16_t* in, float* out, int64_t n, int32_t is_bf16) {
  for (int64_t k = 0; k < n; ++k) out[k] = widen16(in[k], is_bf16);
}

/* ====================================================== building blocks ==== */

float orc_ring_sum(const float* vals, int32_t n_ranks, int32_t owner) {
  /* the chunk starts at rank owner+1 and each rank on the way adds its own
   * value; the last addition is the owner's */
  float acc = vals[(owner + 1) % n_ranks];
  for (int32_t hop = 2; hop <= n_ranks; ++hop) {
    float own = vals[(owner + hop) % n_ranks];
    acc = acc + own;
  }
  return acc;
}

float orc_unscale_factor(float scale, int32_t n_ranks) {
  return orc_unscale_factor_k(scale, n_ranks, 1);
}

float orc_unscale_factor_k(float scale, int32_t n_ranks, int32_t n_micro) {
  double denom = (double)scale * (double)n_ranks;
  denom = denom * (double)n_micro;
  return (float)(1.0 / denom);
}

void orc_accumulate(const uint16_t* micro, float* acc, int64_t n, int32_t is_bf16,
                    int32_t first) {
  for (int64_t k = 0; k < n; ++k) {
    float x = widen16(micro[k], is_bf16);
    acc[k] = first ? x : acc[k] + x;
  }
}

orc_adam_scalars orc_adam_scalars_make(const orc_hparams* hp, int32_t t) {
  orc_adam_scalars a;
  double p1 = 1.0, p2 = 1.0;
  for (int32_t k = 0; k < t; ++k) {
    p1 = p1 * hp->beta1;
    p2 = p2 * hp->beta2;
  }
  a.b1 = (float)hp->beta1;
  a.omb1 = (float)(1.0 - hp->beta1);
  a.b2 = (float)hp->beta2;
  a.omb2 = (float)(1.0 - hp->beta2);
  a.bc1 = (float)(1.0 - p1);
  a.bc2 = (float)(1.0 - p2);
  a.lr = (float)hp->lr;
  double lr_wd = hp->lr * hp->weight_decay;
  a.decay = (float)(1.0 - lr_wd);
  a.eps = (float)hp->eps;
  return a;
}

void orc_adamw_elem(float* theta, float* m, float* v, float g, const orc_adam_scalars* a) {
  /* first moment */
  float m_old = a->b1 * *m;
  float m_new = a->omb1 * g;
  m_new = m_old + m_new;
  /* second moment */
  float gg = g * g;
  float v_old = a->b2 * *v;
  float v_new = a->omb2 * gg;
  v_new = v_old + v_new;
  /* bias corrections */
  float mh = m_new / a->bc1;
  float vh = v_new / a->bc2;
  /* eps outside the square root */
  float den = sqrtf(vh);
  den = den + a->eps;
  float u = mh / den;
  /* decoupled weight decay, then the Adam step */
  float th = *theta * a->decay;
  float step = a->lr * u;
  th = th - step;
  *m = m_new;
  *v = v_new;
  *theta = th;
}

int32_t orc_clip_coef(double norm_sq, double max_norm, float* coef, double* norm) {
  double nrm = sqrt(norm_sq);
  double c = max_norm / (nrm + 1e-6);
  if (norm) *norm = nrm;
  if (c < 1.0) {
    *coef = (float)c;
    return 1;
  }
  *coef = 1.0f;
  return 0;
}

void orc_scaler_finish(orc_scaler* s, const orc_hparams* hp, int32_t overflow) {
  s->overflow = overflow ? 1 : 0;
  if (overflow) {
    if (hp->dynamic_scale) {
      float half = s->scale * 0.5f;
      s->scale = half < 1.0f ? 1.0f : half;
    }
    s->good_steps = 0;
    return;
  }
  s->t = s->t + 1;
  s->good_steps = s->good_steps + 1;
  if (hp->dynamic_scale && s->good_steps >= hp->growth_interval) {
    s->scale = s->scale * 2.0f;
    s->good_steps = 0;
  }
}

/* =========================================================== drivers ==== */

static int64_t bucket_of(const orc_plan* p, int64_t j) {
  return p->bucket_elems == 0 ? 0 : j / p->bucket_elems;
}

/* Replica value of rank r at window index w: 16-bit arrays or fp32 arrays. */
typedef struct replica_reader {
  const uint16_t* const* h16;
  const float* const* f32;
  int32_t is_bf16;
} replica_reader;

static float read_replica(const replica_reader* rd, int32_t r, int64_t w) {
  return rd->f32 ? rd->f32[r][w] : widen16(rd->h16[r][w], rd->is_bf16);
}

static int step_arrays_impl(const orc_plan* p, int32_t rank_lo, int32_t rank_hi,
                            const replica_reader* rd, int32_t n_micro, int32_t is_bf16,
                            int64_t wbase, float* master, float* m, float* v, uint16_t* params,
                            float* ghat, uint32_t* bucket_flags, const orc_hparams* hp,
                            orc_scaler* sc) {
  if (!p || !hp || !sc || n_micro < 1) return -1;
  if (rank_lo < 0 || rank_hi > p->n_ranks || rank_lo > rank_hi) return -1;
  const int32_t N = p->n_ranks;
  const int64_t lo = (int64_t)rank_lo * p->shard;
  const int64_t hi = (int64_t)rank_hi * p->shard;
  if (lo < wbase) return -1;
  const int64_t n = hi - lo;
  float* g = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  float* vals = (float*)malloc((size_t)N * sizeof(float));
  if (!g || !vals) {
    free(g);
    free(vals);
    return -1;
  }
  /* reduce-scatter with unscale and the non-finite check */
  const float inv = orc_unscale_factor_k(sc->scale, N, n_micro);
  int32_t overflow = 0;
  for (int64_t j = lo; j < hi; ++j) {
    int32_t owner = (int32_t)(j / p->shard);
    for (int32_t r = 0; r < N; ++r) vals[r] = read_replica(rd, r, j - wbase);
    float acc = orc_ring_sum(vals, N, owner);
    float gj = acc * inv;
    g[j - lo] = gj;
    if (ghat) ghat[j - wbase] = gj;
    if (!isfinite(gj)) {
      overflow = 1;
      if (bucket_flags) bucket_flags[bucket_of(p, j)] |= 1u;
    }
  }
  if (overflow) {
    orc_scaler_finish(sc, hp, 1);
    free(g);
    free(vals);
    return 0;
  }
  /* optional global-norm clip */
  float coef = 1.0f;
  int32_t apply = 0;
  sc->norm_sq = 0.0;
  sc->norm = 0.0;
  if (hp->max_grad_norm > 0.0) {
    double total = 0.0;
    for (int64_t c0 = 0; c0 < n; c0 += ORC_NORM_CHUNK) {
      double part = 0.0;
      int64_t c1 = imin64(c0 + ORC_NORM_CHUNK, n);
      for (int64_t k = c0; k < c1; ++k) {
        double d = (double)g[k];
        part = part + d * d;
      }
      total = total + part;
    }
    sc->norm_sq = total;
    apply = orc_clip_coef(total, hp->max_grad_norm, &coef, &sc->norm);
  }
  sc->clip_coef = coef;
  /* AdamW on the owned fp32 shard, then the 16-bit working copy */
  orc_adam_scalars a = orc_adam_scalars_make(hp, sc->t + 1);
  for (int64_t j = lo; j < hi; ++j) {
    float gj = g[j - lo];
    if (apply) gj = gj * coef;
    int64_t w = j - wbase;
    orc_adamw_elem(&master[w], &m[w], &v[w], gj, &a);
    params[w] = cast16(master[w], is_bf16);
  }
  orc_scaler_finish(sc, hp, 0);
  free(g);
  free(vals);
  return 0;
}

int orc_step_arrays(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, int32_t is_bf16,
                    const uint16_t* const* replicas, int64_t wbase, float* master,
                    float* m, float* v, uint16_t* params, float* ghat,
                    uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc) {
  if (!replicas) return -1;
  replica_reader rd = {replicas, NULL, is_bf16};
  return step_arrays_impl(p, rank_lo, rank_hi, &rd, 1, is_bf16, wbase, master, m, v, params,
                          ghat, bucket_flags, hp, sc);
}

int orc_step_arrays_f32(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, int32_t is_bf16,
                        const float* const* replicas, int32_t n_micro, int64_t wbase,
                        float* master, float* m, float* v, uint16_t* params, float* ghat,
                        uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc) {
  if (!replicas) return -1;
  replica_reader rd = {NULL, replicas, is_bf16};
  return step_arrays_impl(p, rank_lo, rank_hi, &rd, n_micro, is_bf16, wbase, master, m, v,
                          params, ghat, bucket_flags, hp, sc);
}

/* ---------------------------------------------- generator-driven driver ---- */

/* Replica value of flat element j for every rank, widened to fp32. The
 * per-(step, rank) generator streams are formed once per call site. */
static float gen_value(const orc_gen* g, const zs_grad_stream* st, uint32_t step, int32_t rank,
                       int64_t j) {
  uint16_t bits;
  if (g->inject_step >= 0 && (uint32_t)g->inject_step == step && g->inject_rank == rank &&
      g->inject_elem == j) {
    bits = (uint16_t)g->inject_bits;
  } else {
    bits = cast16(zs_grad_stream_value(st, j), g->is_bf16);
  }
  return widen16(bits, g->is_bf16);
}

static zs_grad_stream* make_streams(const orc_plan* p, const orc_gen* g, float scale,
                                    uint32_t step) {
  zs_grad_stream* st = (zs_grad_stream*)malloc((size_t)p->n_ranks * sizeof(zs_grad_stream));
  if (!st) return NULL;
  zs_grad_spec spec = g->spec;
  spec.loss_scale = scale;
  for (int32_t r = 0; r < p->n_ranks; ++r) st[r] = zs_grad_stream_make(&spec, step, (uint32_t)r);
  return st;
}

static float gen_ghat(const orc_plan* p, const orc_gen* g, const zs_grad_stream* st, float inv,
                      uint32_t step, int64_t j, float* vals) {
  int32_t N = p->n_ranks;
  for (int32_t r = 0; r < N; ++r) vals[r] = gen_value(g, &st[r], step, r, j);
  float acc = orc_ring_sum(vals, N, (int32_t)(j / p->shard));
  return acc * inv;
}

typedef struct pass_job {
  const orc_plan* p;
  const orc_gen* g;
  const zs_grad_stream* st;
  uint32_t step;
  float inv;
  int64_t lo, hi, n_chunks;
  int32_t worker, n_workers;
  double* chunk_sq;         /* per chunk */
  int32_t* chunk_bad;       /* per chunk */
  uint32_t* flags;          /* per worker: n_buckets words */
} pass_job;

static void* pass_worker(void* arg) {
  pass_job* J = (pass_job*)arg;
  const orc_plan* p = J->p;
  float* vals = (float*)malloc((size_t)p->n_ranks * sizeof(float));
  uint32_t* flags = J->flags + (size_t)J->worker * (size_t)(p->n_buckets > 0 ? p->n_buckets : 1);
  for (int64_t c = J->worker; c < J->n_chunks; c += J->n_workers) {
    int64_t a = J->lo + c * ORC_NORM_CHUNK;
    int64_t b = imin64(a + ORC_NORM_CHUNK, J->hi);
    double part = 0.0;
    int32_t bad = 0;
    for (int64_t j = a; j < b; ++j) {
      float gj = gen_ghat(p, J->g, J->st, J->inv, J->step, j, vals);
      if (!isfinite(gj)) {
        bad = 1;
        flags[bucket_of(p, j)] |= 1u;
      }
      double d = (double)gj;
      part = part + d * d;
    }
    J->chunk_sq[c] = part;
    J->chunk_bad[c] = bad;
  }
  free(vals);
  return NULL;
}

int orc_gen_step(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, const orc_gen* g,
                 uint32_t step, int32_t n_threads, const int64_t* elems, int64_t n_elems,
                 float* master, float* m, float* v, uint16_t* params,
                 uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc) {
  if (!p || !g || !hp || !sc) return -1;
  if (rank_lo < 0 || rank_hi > p->n_ranks || rank_lo > rank_hi) return -1;
  if (n_threads < 1) n_threads = 1;
  const int64_t lo = (int64_t)rank_lo * p->shard;
  const int64_t hi = (int64_t)rank_hi * p->shard;
  const int64_t n_chunks = (hi - lo + ORC_NORM_CHUNK - 1) / ORC_NORM_CHUNK;
  const int32_t nb = p->n_buckets > 0 ? p->n_buckets : 1;
  double* chunk_sq = (double*)calloc((size_t)(n_chunks > 0 ? n_chunks : 1), sizeof(double));
  int32_t* chunk_bad = (int32_t*)calloc((size_t)(n_chunks > 0 ? n_chunks : 1), sizeof(int32_t));
  uint32_t* wflags = (uint32_t*)calloc((size_t)n_threads * (size_t)nb, sizeof(uint32_t));
  pass_job* jobs = (pass_job*)calloc((size_t)n_threads, sizeof(pass_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  float* vals = (float*)malloc((size_t)p->n_ranks * sizeof(float));
  zs_grad_stream* streams = NULL;
  int rc = 0;
  if (!chunk_sq || !chunk_bad || !wflags || !jobs || !th || !vals) {
    rc = -1;
    goto done;
  }
  const float inv = orc_unscale_factor(sc->scale, p->n_ranks);
  streams = make_streams(p, g, sc->scale, step);
  if (!streams) {
    rc = -1;
    goto done;
  }
  for (int32_t w = 0; w < n_threads; ++w) {
    pass_job J = {p, g, streams, step, inv, lo, hi, n_chunks, w, n_threads, chunk_sq, chunk_bad, wflags};
    jobs[w] = J;
  }
  for (int32_t w = 1; w < n_threads; ++w) pthread_create(&th[w], NULL, pass_worker, &jobs[w]);
  pass_worker(&jobs[0]);
  for (int32_t w = 1; w < n_threads; ++w) pthread_join(th[w], NULL);

  int32_t overflow = 0;
  double total = 0.0;
  for (int64_t c = 0; c < n_chunks; ++c) {
    overflow |= chunk_bad[c];
    total = total + chunk_sq[c];
  }
  if (bucket_flags)
    for (int32_t w = 0; w < n_threads; ++w)
      for (int32_t k = 0; k < p->n_buckets; ++k) bucket_flags[k] |= wflags[(size_t)w * nb + k];
  if (overflow) {
    orc_scaler_finish(sc, hp, 1);
    goto done;
  }
  float coef = 1.0f;
  int32_t apply = 0;
  sc->norm_sq = 0.0;
  sc->norm = 0.0;
  if (hp->max_grad_norm > 0.0) {
    sc->norm_sq = total;
    apply = orc_clip_coef(total, hp->max_grad_norm, &coef, &sc->norm);
  }
  sc->clip_coef = coef;
  orc_adam_scalars a = orc_adam_scalars_make(hp, sc->t + 1);
  for (int64_t k = 0; k < n_elems; ++k) {
    int64_t j = elems[k];
    if (j < lo || j >= hi) {
      rc = -1;
      goto done;
    }
    float gj = gen_ghat(p, g, streams, inv, step, j, vals);
    if (apply) gj = gj * coef;
    orc_adamw_elem(&master[k], &m[k], &v[k], gj, &a);
    params[k] = cast16(master[k], g->is_bf16);
  }
  orc_scaler_finish(sc, hp, 0);
done:
  free(chunk_sq);
  free(chunk_bad);
  free(wflags);
  free(jobs);
  free(th);
  free(vals);
  free(streams);
  return rc;
}

int orc_gen_ghat(const orc_plan* p, const orc_gen* g, uint32_t step, float scale,
                 const int64_t* elems, int64_t n_elems, float* ghat) {
  if (!p || !g || !ghat) return -1;
  float* vals = (float*)malloc((size_t)p->n_ranks * sizeof(float));
  zs_grad_stream* st = make_streams(p, g, scale, step);
  if (!vals || !st) {
    free(vals);
    free(st);
    return -1;
  }
  const float inv = orc_unscale_factor(scale, p->n_ranks);
  for (int64_t k = 0; k < n_elems; ++k) ghat[k] = gen_ghat(p, g, st, inv, step, elems[k], vals);
  free(vals);
  free(st);
  return 0;
}
