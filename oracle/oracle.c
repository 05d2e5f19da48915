/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow fp64 CPU statement of the Flux-style attention call:
 *     O = softmax(scale * RoPE(RMSNorm_q(q)) RoPE(RMSNorm_k(k))^T + mask) V
 * and its gradients. Every step materialises its full intermediate (the whole
 * S_q x S_kv score, probability and gradient matrices of a head); nothing is
 * tiled, fused or reordered. It shares no code with the CUDA library and is
 * only ever loaded by the test-suite, by the smoke check and by the benchmark's
 * CPU-baseline leg.
 *
 * Sources (page titles and sections):
 *  - "Flux-family attention: flash-attn and other backends fail in an autocast
 *    context" (diffusers issue 14104), "Root cause" list: q and k pass through
 *    norm_q / norm_k (torch.nn.RMSNorm over the head dimension), then the
 *    rotary embedding, then attention; v goes straight to attention.
 *  - "Metal Flash Attention" (SimpleTuner docs), section "Fused RoPE + SDPA":
 *    interleaved-pair rotation of Q and K, one angle per pair (pair-duplicated
 *    cos/sin tables), gradients returned w.r.t. the pre-RoPE Q/K through the
 *    inverse rotation (the same rotation with sin negated).
 *  - same page, section "Enable In SimpleTuner": bool masks (True = attend),
 *    additive float masks, batched [B,H,S_q,S_kv] and broadcast [B,1,1,S_kv]
 *    masks; causal calls.
 * Readings where the pages are silent (frequency formula, rotation sign,
 * fully-masked rows, causal alignment) are stated beside the code below.
 *
 * Layouts: q, dq, o, do are [B, S_q, H, D]; k, v, dk, dv are [B, S_kv, H_kv, D]
 * with H a multiple of H_kv; all contiguous fp64. Grouped K/V heads (same page,
 * section "Fused RoPE + SDPA": GQA inputs are rotated at the K/V head count and
 * expanded afterwards): query head h attends with K/V head h / (H / H_kv), and
 * dk, dv of a K/V head sum the gradients of its group of query heads. The rotation comes either from angles phi [Bp, S, D/2]
 * or from the pages' cos/sin tables [Bp, S, D] (same page, section "Fused
 * RoPE + SDPA": pair-duplicated tables of shape [S, D], [1, S, D] or
 * [B, S, D]), with Bp in {1, B}.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Multi-axis rotary angles ("Fused RoPE + SDPA": one angle per interleaved
 * pair). Reading: axis a owns head dims [o_a, o_a + d_a) with o_a the sum of
 * the earlier axes' widths; inside axis a, pair j (dims o_a+2j, o_a+2j+1) has
 * frequency theta^(-2j/d_a), j restarting at 0 in every axis, and angle
 * id[a] * frequency.
 *   ids: [n_tok, n_axes] (position ids of each token), phi: [n_tok, D/2]. */
void oracle_rope_angles(const double* ids, int64_t n_tok, int n_axes, const int* axes_dim, double theta,
                        double* phi) {
  int D = 0;
  for (int a = 0; a < n_axes; ++a) D += axes_dim[a];
  for (int64_t t = 0; t < n_tok; ++t) {
    int pair = 0;
    for (int a = 0; a < n_axes; ++a) {
      const int d_a = axes_dim[a];
      for (int j = 0; j < d_a / 2; ++j) {
        const double freq = pow(theta, -2.0 * (double)j / (double)d_a);
        phi[t * (D / 2) + pair] = ids[t * n_axes + a] * freq;
        ++pair;
      }
    }
  }
}

/* RMSNorm of one row (torch.nn.RMSNorm over the head dimension, eps inside
 * the square root): r = 1/sqrt(mean(x^2) + eps), y = x * r * w. */
static double rmsnorm_row(const double* x, const double* w, int D, double eps, double* y) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += x[d] * x[d];
  const double r = 1.0 / sqrt(ss / (double)D + eps);
  for (int d = 0; d < D; ++d) y[d] = x[d] * r * w[d];
  return r;
}

/* Rotation source of one head: angles (phi: [S][D/2]) or the pages' tables
 * (cos, sin: [S][D]); exactly one of phi and cos is set. */
typedef struct {
  const double* phi;
  const double* cos;
  const double* sin;
} rot_src;

/* The rows of batch element b (per-sample sources have Bp = B). */
static rot_src rot_at(const rot_src* r, int bp, int b, int S, int D) {
  const int64_t bi = bp > 1 ? b : 0;
  rot_src o = {NULL, NULL, NULL};
  if (r->phi) o.phi = r->phi + bi * S * (D / 2);
  else {
    o.cos = r->cos + bi * S * D;
    o.sin = r->sin + bi * S * D;
  }
  return o;
}

/* Interleaved-pair rotation (counter-clockwise) of row s:
 *   angles: y0 = x0 cos(phi) - x1 sin(phi),  y1 = x0 sin(phi) + x1 cos(phi);
 *   tables: y = x * cos + rot(x) * sin elementwise, rot(x) = (-x1, x0) per
 *   pair, which is the same rotation when the tables are pair-duplicated. */
static void rope_row(const double* x, const rot_src* r, int64_t s, int D, double* y) {
  for (int p = 0; p < D / 2; ++p) {
    if (r->phi) {
      const double c = cos(r->phi[s * (D / 2) + p]), sn = sin(r->phi[s * (D / 2) + p]);
      y[2 * p] = x[2 * p] * c - x[2 * p + 1] * sn;
      y[2 * p + 1] = x[2 * p] * sn + x[2 * p + 1] * c;
    } else {
      const double* c = r->cos + s * D + 2 * p;
      const double* sn = r->sin + s * D + 2 * p;
      y[2 * p] = x[2 * p] * c[0] - x[2 * p + 1] * sn[0];
      y[2 * p + 1] = x[2 * p + 1] * c[1] + x[2 * p] * sn[1];
    }
  }
}

/* Transpose of that rotation (the backward): for angles, the same pairwise
 * rotation with sin negated; for tables, the transpose of the elementwise form
 * (equal to it when the tables are pair-duplicated). */
static void rope_row_inverse(const double* g, const rot_src* r, int64_t s, int D, double* y) {
  for (int p = 0; p < D / 2; ++p) {
    if (r->phi) {
      const double c = cos(r->phi[s * (D / 2) + p]), sn = -sin(r->phi[s * (D / 2) + p]);
      y[2 * p] = g[2 * p] * c - g[2 * p + 1] * sn;
      y[2 * p + 1] = g[2 * p] * sn + g[2 * p + 1] * c;
    } else {
      const double* c = r->cos + s * D + 2 * p;
      const double* sn = r->sin + s * D + 2 * p;
      y[2 * p] = g[2 * p] * c[0] + g[2 * p + 1] * sn[1];
      y[2 * p + 1] = g[2 * p + 1] * c[1] - g[2 * p] * sn[0];
    }
  }
}

/* Pre-attention transform of one head: out[s][:] = RoPE(RMSNorm(x[b,s,h,:])).
 * r_out[s] receives the RMSNorm reciprocal root of each row. */
static void transform_head(const double* x, int S, int H, int D, int b, int h, const double* w, double eps,
                           const rot_src* rot, double* out, double* r_out) {
#pragma omp parallel for schedule(static)
  for (int s = 0; s < S; ++s) {
    double tmp[1024];
    const double* xr = x + (((int64_t)b * S + s) * H + h) * D;
    r_out[s] = rmsnorm_row(xr, w, D, eps, tmp);
    rope_row(tmp, rot, s, D, out + (int64_t)s * D);
  }
}

/* Exported for the pins: rows x [n_rows][D] -> RoPE(RMSNorm(x)) with one
 * angle row phi [n_rows][D/2] per input row. */
void oracle_qk_transform(const double* x, int64_t n_rows, int D, const double* w, double eps, const double* phi,
                         double* out) {
  const rot_src rot = {phi, NULL, NULL};
  for (int64_t s = 0; s < n_rows; ++s) {
    double tmp[1024];
    rmsnorm_row(x + s * D, w, D, eps, tmp);
    rope_row(tmp, &rot, s, D, out + s * D);
  }
}

/* As oracle_qk_transform with the pages' tables: cos, sin [n_rows][D]. */
void oracle_qk_transform_tab(const double* x, int64_t n_rows, int D, const double* w, double eps,
                             const double* cos_t, const double* sin_t, double* out) {
  const rot_src rot = {NULL, cos_t, sin_t};
  for (int64_t s = 0; s < n_rows; ++s) {
    double tmp[1024];
    rmsnorm_row(x + s * D, w, D, eps, tmp);
    rope_row(tmp, &rot, s, D, out + s * D);
  }
}

/* Mask value at (b, h, i, j): returns 0 for "attend unchanged", -inf for a
 * bool False, or the additive value. kind: 0 none, 1 bool (uint8), 2 additive. */
static double mask_value(int kind, const void* mask, const int64_t* ms, int b, int h, int i, int j) {
  if (kind == 0) return 0.0;
  const int64_t off = (int64_t)b * ms[0] + (int64_t)h * ms[1] + (int64_t)i * ms[2] + (int64_t)j * ms[3];
  if (kind == 1) return ((const uint8_t*)mask)[off] ? 0.0 : -INFINITY;
  return ((const double*)mask)[off];
}

/* Scores and probabilities of one head, both [Sq][Skv]:
 *   s_ij = scale * q'_i . k'_j + mask_ij   (-inf where a bool mask is False
 *          or, when causal, where j > i — top-left aligned, as torch's
 *          is_causal);
 *   P = row softmax, lse_i = ln sum_j exp(s_ij).
 * A row whose every entry is -inf gets P = 0 and lse = -inf (reading: the
 * pages define no output there; zero output, zero gradient). */
static void head_probs(const double* qp, const double* kp, int Sq, int Skv, int D, double scale, int kind,
                       const void* mask, const int64_t* ms, int causal, int b, int h, double* P, double* lse) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < Sq; ++i) {
    double* row = P + (int64_t)i * Skv;
    double m = -INFINITY;
    for (int j = 0; j < Skv; ++j) {
      double s = 0.0;
      for (int d = 0; d < D; ++d) s += qp[(int64_t)i * D + d] * kp[(int64_t)j * D + d];
      s = scale * s + mask_value(kind, mask, ms, b, h, i, j);
      if (causal && j > i) s = -INFINITY;
      row[j] = s;
      if (s > m) m = s;
    }
    if (m == -INFINITY) {
      for (int j = 0; j < Skv; ++j) row[j] = 0.0;
      lse[i] = -INFINITY;
      continue;
    }
    double l = 0.0;
    for (int j = 0; j < Skv; ++j) {
      row[j] = exp(row[j] - m);
      l += row[j];
    }
    for (int j = 0; j < Skv; ++j) row[j] /= l;
    lse[i] = m + log(l);
  }
}

/* out[r][:] = sum_c M[r][c] * Y[c][:]   (M is [R][C], Y is [C][D]) */
static void mat_ab(const double* M, int R, int C, const double* Y, int D, double* out) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < R; ++r) {
    double* o = out + (int64_t)r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int c = 0; c < C; ++c) {
      const double a = M[(int64_t)r * C + c];
      if (a == 0.0) continue;
      for (int d = 0; d < D; ++d) o[d] += a * Y[(int64_t)c * D + d];
    }
  }
}

/* out[c][:] = sum_r M[r][c] * X[r][:]   (M is [R][C], X is [R][D]) */
static void mat_atb(const double* M, int R, int C, const double* X, int D, double* out) {
#pragma omp parallel for schedule(static)
  for (int c = 0; c < C; ++c) {
    double* o = out + (int64_t)c * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int r = 0; r < R; ++r) {
      const double a = M[(int64_t)r * C + c];
      if (a == 0.0) continue;
      for (int d = 0; d < D; ++d) o[d] += a * X[(int64_t)r * D + d];
    }
  }
}

/* Copy head h of batch b of x [B,S,H,D] into a [S][D] matrix. */
static void gather_head(const double* x, int S, int H, int D, int b, int h, double* out) {
  for (int s = 0; s < S; ++s)
    memcpy(out + (int64_t)s * D, x + (((int64_t)b * S + s) * H + h) * D, sizeof(double) * D);
}
static void scatter_head(const double* m, int S, int H, int D, int b, int h, double* x) {
  for (int s = 0; s < S; ++s)
    memcpy(x + (((int64_t)b * S + s) * H + h) * D, m + (int64_t)s * D, sizeof(double) * D);
}
static void add_head(const double* m, int S, int H, int D, int b, int h, double* x) {
  for (int s = 0; s < S; ++s)
    for (int d = 0; d < D; ++d) x[(((int64_t)b * S + s) * H + h) * D + d] += m[(int64_t)s * D + d];
}
static void zero_head(int S, int H, int D, int b, int h, double* x) {
  for (int s = 0; s < S; ++s) memset(x + (((int64_t)b * S + s) * H + h) * D, 0, sizeof(double) * D);
}

/* Forward for the heads listed in `bh` (flattened b*H + h; NULL = all).
 * rot_q: Bpq x Sq rows, rot_k: Bpk x Skv rows (Bp* in {1, B}).
 * Writes o [B,Sq,H,D] and lse [B,H,Sq] at the listed heads only.
 * Returns 0, or -1 when a work buffer cannot be allocated. */
static int fwd_impl(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
                    const double* wq, const double* wk, double eps, rot_src rot_q, int bpq, rot_src rot_k, int bpk,
                    int mask_kind, const void* mask, const int64_t* mask_strides, int causal, double scale,
                    const int* bh, int n_bh, double* o, double* lse) {
  double* qp = malloc(sizeof(double) * (size_t)Sq * D);
  double* kp = malloc(sizeof(double) * (size_t)Skv * D);
  double* vh = malloc(sizeof(double) * (size_t)Skv * D);
  double* oh = malloc(sizeof(double) * (size_t)Sq * D);
  double* rq = malloc(sizeof(double) * (size_t)Sq);
  double* rk = malloc(sizeof(double) * (size_t)Skv);
  double* P = malloc(sizeof(double) * (size_t)Sq * Skv);
  int rc = 0;
  if (!qp || !kp || !vh || !oh || !rq || !rk || !P) { rc = -1; goto done; }
  const int n = bh ? n_bh : B * H;
  for (int t = 0; t < n; ++t) {
    const int idx = bh ? bh[t] : t;
    const int b = idx / H, h = idx % H;
    const int hk = h / (H / Hkv);  /* the K/V head of query head h */
    const rot_src rq_b = rot_at(&rot_q, bpq, b, Sq, D), rk_b = rot_at(&rot_k, bpk, b, Skv, D);
    transform_head(q, Sq, H, D, b, h, wq, eps, &rq_b, qp, rq);
    transform_head(k, Skv, Hkv, D, b, hk, wk, eps, &rk_b, kp, rk);
    gather_head(v, Skv, Hkv, D, b, hk, vh);
    head_probs(qp, kp, Sq, Skv, D, scale, mask_kind, mask, mask_strides, causal, b, h, P,
               lse + ((int64_t)b * H + h) * Sq);
    mat_ab(P, Sq, Skv, vh, D, oh);
    scatter_head(oh, Sq, H, D, b, h, o);
  }
done:
  free(qp); free(kp); free(vh); free(oh); free(rq); free(rk); free(P);
  return rc;
}

/* Forward with angles: phi_q [Bpq, Sq, D/2], phi_k [Bpk, Skv, D/2]. */
int oracle_fwd(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
               const double* wq, const double* wk, double eps, const double* phi_q, int bpq, const double* phi_k,
               int bpk, int mask_kind, const void* mask, const int64_t* mask_strides, int causal, double scale,
               const int* bh, int n_bh, double* o, double* lse) {
  const rot_src rq = {phi_q, NULL, NULL}, rk = {phi_k, NULL, NULL};
  return fwd_impl(B, Sq, Skv, H, Hkv, D, q, k, v, wq, wk, eps, rq, bpq, rk, bpk, mask_kind, mask, mask_strides, causal,
                  scale, bh, n_bh, o, lse);
}

/* Forward with the pages' tables: cos_q, sin_q [Bpq, Sq, D]; cos_k, sin_k [Bpk, Skv, D]. */
int oracle_fwd_tab(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
                   const double* wq, const double* wk, double eps, const double* cos_q, const double* sin_q, int bpq,
                   const double* cos_k, const double* sin_k, int bpk, int mask_kind, const void* mask,
                   const int64_t* mask_strides, int causal, double scale, const int* bh, int n_bh, double* o,
                   double* lse) {
  const rot_src rq = {NULL, cos_q, sin_q}, rk = {NULL, cos_k, sin_k};
  return fwd_impl(B, Sq, Skv, H, Hkv, D, q, k, v, wq, wk, eps, rq, bpq, rk, bpk, mask_kind, mask, mask_strides, causal,
                  scale, bh, n_bh, o, lse);
}

/* RMSNorm + RoPE backward of one head. gp: gradient w.r.t. the rotated,
 * normalised rows [S][D]; x: raw input [B,S,H,D]. Adds dx into [B,S,H,D]
 * and sum_s (R^T gp) * x * r into dw.
 *   dy = R^T gp (inverse rotation), g = w * dy,
 *   dx = r g - (r^3 / D) x (x . g),   dw += dy * x * r. */
static void transform_head_bwd(const double* gp, const double* x, int S, int H, int D, int b, int h,
                               const double* w, const rot_src* rot, const double* r, double* dx, double* dw) {
  /* dx is added to (the rows start at zero), so that the query heads of a
   * K/V group sum into their K/V head's rows */
  double* dy_all = malloc(sizeof(double) * (size_t)S * D);
#pragma omp parallel for schedule(static)
  for (int s = 0; s < S; ++s) {
    double g[1024];
    double* dy = dy_all + (int64_t)s * D;
    const double* xr = x + (((int64_t)b * S + s) * H + h) * D;
    double* dxr = dx + (((int64_t)b * S + s) * H + h) * D;
    rope_row_inverse(gp + (int64_t)s * D, rot, s, D, dy);
    double xg = 0.0;
    for (int d = 0; d < D; ++d) {
      g[d] = w[d] * dy[d];
      xg += xr[d] * g[d];
    }
    const double rs = r[s];
    for (int d = 0; d < D; ++d) dxr[d] += rs * g[d] - (rs * rs * rs / (double)D) * xr[d] * xg;
  }
  for (int s = 0; s < S; ++s) {
    const double* xr = x + (((int64_t)b * S + s) * H + h) * D;
    for (int d = 0; d < D; ++d) dw[d] += dy_all[(int64_t)s * D + d] * xr[d] * r[s];
  }
  free(dy_all);
}

/* Backward for the listed heads, given dO [B,Sq,H,D]:
 *   dV = P^T dO, dP = dO V^T, Delta_i = sum_j P_ij dP_ij, dS = P (dP - Delta),
 *   dQ' = scale dS K', dK' = scale dS^T Q', then the RoPE/RMSNorm backward.
 * dwq/dwk [D] receive the sums over the listed heads only, and dk/dv of a K/V
 * head the sums over the listed query heads of its group.
 * Returns 0, or -1 when a work buffer cannot be allocated. */
static int bwd_impl(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
                    const double* wq, const double* wk, double eps, rot_src rot_q, int bpq, rot_src rot_k, int bpk,
                    int mask_kind, const void* mask, const int64_t* mask_strides, int causal, double scale,
                    const double* dout, const int* bh, int n_bh, double* dq, double* dk, double* dv, double* dwq,
                    double* dwk) {
  double* qp = malloc(sizeof(double) * (size_t)Sq * D);
  double* kp = malloc(sizeof(double) * (size_t)Skv * D);
  double* vh = malloc(sizeof(double) * (size_t)Skv * D);
  double* doh = malloc(sizeof(double) * (size_t)Sq * D);
  double* rq = malloc(sizeof(double) * (size_t)Sq);
  double* rk = malloc(sizeof(double) * (size_t)Skv);
  double* lse = malloc(sizeof(double) * (size_t)Sq);
  double* P = malloc(sizeof(double) * (size_t)Sq * Skv);
  double* dS = malloc(sizeof(double) * (size_t)Sq * Skv);
  double* dvh = malloc(sizeof(double) * (size_t)Skv * D);
  double* gq = malloc(sizeof(double) * (size_t)Sq * D);
  double* gk = malloc(sizeof(double) * (size_t)Skv * D);
  int rc = 0;
  if (!qp || !kp || !vh || !doh || !rq || !rk || !lse || !P || !dS || !dvh || !gq || !gk) { rc = -1; goto done; }
  for (int d = 0; d < D; ++d) { dwq[d] = 0.0; dwk[d] = 0.0; }
  const int n = bh ? n_bh : B * H;
  for (int t = 0; t < n; ++t) { /* the gradient rows of the listed heads start at zero */
    const int idx = bh ? bh[t] : t;
    const int b = idx / H, h = idx % H, hk = h / (H / Hkv);
    zero_head(Sq, H, D, b, h, dq);
    zero_head(Skv, Hkv, D, b, hk, dk);
    zero_head(Skv, Hkv, D, b, hk, dv);
  }
  for (int t = 0; t < n; ++t) {
    const int idx = bh ? bh[t] : t;
    const int b = idx / H, h = idx % H;
    const int hk = h / (H / Hkv);  /* the K/V head of query head h */
    const rot_src pq = rot_at(&rot_q, bpq, b, Sq, D), pk = rot_at(&rot_k, bpk, b, Skv, D);
    transform_head(q, Sq, H, D, b, h, wq, eps, &pq, qp, rq);
    transform_head(k, Skv, Hkv, D, b, hk, wk, eps, &pk, kp, rk);
    gather_head(v, Skv, Hkv, D, b, hk, vh);
    gather_head(dout, Sq, H, D, b, h, doh);
    head_probs(qp, kp, Sq, Skv, D, scale, mask_kind, mask, mask_strides, causal, b, h, P, lse);
    /* dV = P^T dO */
    mat_atb(P, Sq, Skv, doh, D, dvh);
    add_head(dvh, Skv, Hkv, D, b, hk, dv);
    /* dP = dO V^T, Delta, dS = P (dP - Delta) */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Sq; ++i) {
      double delta = 0.0;
      for (int j = 0; j < Skv; ++j) {
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += doh[(int64_t)i * D + d] * vh[(int64_t)j * D + d];
        dS[(int64_t)i * Skv + j] = dp;
        delta += P[(int64_t)i * Skv + j] * dp;
      }
      for (int j = 0; j < Skv; ++j) {
        const int64_t ij = (int64_t)i * Skv + j;
        dS[ij] = P[ij] * (dS[ij] - delta);
      }
    }
    /* dQ' = scale dS K', dK' = scale dS^T Q' */
    mat_ab(dS, Sq, Skv, kp, D, gq);
    mat_atb(dS, Sq, Skv, qp, D, gk);
    for (int64_t e = 0; e < (int64_t)Sq * D; ++e) gq[e] *= scale;
    for (int64_t e = 0; e < (int64_t)Skv * D; ++e) gk[e] *= scale;
    transform_head_bwd(gq, q, Sq, H, D, b, h, wq, &pq, rq, dq, dwq);
    transform_head_bwd(gk, k, Skv, Hkv, D, b, hk, wk, &pk, rk, dk, dwk);
  }
done:
  free(qp); free(kp); free(vh); free(doh); free(rq); free(rk); free(lse);
  free(P); free(dS); free(dvh); free(gq); free(gk);
  return rc;
}

/* Backward with angles: phi_q [Bpq, Sq, D/2], phi_k [Bpk, Skv, D/2]. */
int oracle_bwd(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
               const double* wq, const double* wk, double eps, const double* phi_q, int bpq, const double* phi_k,
               int bpk, int mask_kind, const void* mask, const int64_t* mask_strides, int causal, double scale,
               const double* dout, const int* bh, int n_bh, double* dq, double* dk, double* dv, double* dwq,
               double* dwk) {
  const rot_src rq = {phi_q, NULL, NULL}, rk = {phi_k, NULL, NULL};
  return bwd_impl(B, Sq, Skv, H, Hkv, D, q, k, v, wq, wk, eps, rq, bpq, rk, bpk, mask_kind, mask, mask_strides, causal,
                  scale, dout, bh, n_bh, dq, dk, dv, dwq, dwk);
}

/* Backward with the pages' tables: cos_q, sin_q [Bpq, Sq, D]; cos_k, sin_k [Bpk, Skv, D]. */
int oracle_bwd_tab(int B, int Sq, int Skv, int H, int Hkv, int D, const double* q, const double* k, const double* v,
                   const double* wq, const double* wk, double eps, const double* cos_q, const double* sin_q, int bpq,
                   const double* cos_k, const double* sin_k, int bpk, int mask_kind, const void* mask,
                   const int64_t* mask_strides, int causal, double scale, const double* dout, const int* bh, int n_bh,
                   double* dq, double* dk, double* dv, double* dwq, double* dwk) {
  const rot_src rq = {NULL, cos_q, sin_q}, rk = {NULL, cos_k, sin_k};
  return bwd_impl(B, Sq, Skv, H, Hkv, D, q, k, v, wq, wk, eps, rq, bpq, rk, bpk, mask_kind, mask, mask_strides, causal,
                  scale, dout, bh, n_bh, dq, dk, dv, dwq, dwk);
}
