// The exact-fp32 path: q, k, v (and dO) all fp32, every product and sum in
// fp32 on the CUDA cores ("Metal Flash Attention", section "Requirements":
// FP32 runs natively there, the parity probe of section "Synthetic Memory
// Probe" is an FP32 run). The tensor-core kernels round their operands to
// 16 bits, which no fp32 tolerance admits; these kernels trade speed for
// fp32 results.
//
// Tiles of 64 rows x D = 128, 256 threads. Shared-memory rows are 129 floats
// apart, so that a warp walking a column (16 rows at a stride of 129) and a
// warp walking a row hit 16 or 32 different banks. Thread (ty, tx) = (tid/16,
// tid%16) owns rows ty + 16 i (i < 4) and columns tx + 16 j of every product.
//   forward  (query tile, head, batch): S = Q' K'^T, online base-2 softmax,
//            O += P V, then O / l and the log-sum-exp;
//   dK / dV  (key tile, K/V head, batch): over every query tile of every
//            query head of the K/V group, recompute P from the LSE, dP = dO V^T,
//            dS = P (dP - Delta), dV += P^T dO, dK' += dS^T Q'; then the
//            inverse rotation and the RMSNorm backward of each key row;
//   dQ       (query tile, head, batch): over the key tiles, dQ' += dS K'; then
//            the same row transform for the query rows.
// Q' / K' are RMSNorm + rotation of the raw rows, computed in fp32 when a tile
// is loaded. No atomics: dk, dv, dq and the norm-weight partials are written
// once, in a fixed order.
#include "st_common.cuh"
#include "st_f32.h"
#include "st_kernels.h"

namespace st {

namespace {

constexpr int kT = 64;                 // rows per tile
constexpr int kLd = kD + 1;            // row stride of the [64][D] tiles (floats)
constexpr int kLdP = kT + 1;           // row stride of the [64][64] tiles
constexpr int kThreads = 256;
constexpr uint32_t kTileF = kT * kLd;  // floats per [64][D] tile
constexpr uint32_t kTileP = kT * kLdP;
constexpr uint32_t kFwdSmemF = (3 * kTileF + kTileP) * 4;
constexpr uint32_t kBwdKVSmemF = (4 * kTileF + 2 * kTileP) * 4;
constexpr uint32_t kBwdQSmemF = (4 * kTileF + kTileP) * 4;

__device__ __forceinline__ int tiles64(int n) { return (n + kT - 1) / kT; }

// Rows row0 .. row0 + 63 of x (head h, batch b) into dst: RMSNorm in fp32
// (weight w) and the interleaved-pair rotation by the (cos, sin) rows of tab;
// rows at or past nrows become zeros. Four threads per row, 32 dims each.
__device__ __forceinline__ void load_rot(float* dst, const RowTensor& x, int b, int h, int row0, int nrows,
                                         const float2* tab, const float* w, float eps) {
  const int r = threadIdx.x >> 2, part = threadIdx.x & 3, row = row0 + r;
  const bool ok = row < nrows;
  float v[32];
  const int64_t off = b * x.sb + (int64_t)(ok ? row : 0) * x.ss + h * x.sh;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float x8[8];
    if (ok) {
      load_chunk8(x.p, off, x.dt, 4 * part + c, x8);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x8[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[8 * c + e] = x8[e];
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const float rr = rsqrtf(ss * (1.0f / kD) + eps);
  const float2* t = tab + (int64_t)(ok ? row : 0) * kPairs + 16 * part;
  float* out = dst + r * kLd + 32 * part;
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const float2 cs = ok ? t[p] : make_float2(1.f, 0.f);
    const float n0 = v[2 * p] * w[32 * part + 2 * p] * rr, n1 = v[2 * p + 1] * w[32 * part + 2 * p + 1] * rr;
    out[2 * p] = n0 * cs.x - n1 * cs.y;
    out[2 * p + 1] = n0 * cs.y + n1 * cs.x;
  }
}

// Rows row0 .. row0 + 63 of an fp32 [B, S, H, D] tensor into dst (zeros past nrows).
__device__ __forceinline__ void load_plain(float* dst, const float* base, int64_t sb, int64_t ss, int64_t sh, int b,
                                           int h, int row0, int nrows) {
  const int r = threadIdx.x >> 2, part = threadIdx.x & 3, row = row0 + r;
  const float4* src = reinterpret_cast<const float4*>(base + b * sb + (int64_t)row * ss + h * sh) + 8 * part;
  float* out = dst + r * kLd + 32 * part;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 a = row < nrows ? __ldg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    out[4 * c] = a.x;
    out[4 * c + 1] = a.y;
    out[4 * c + 2] = a.z;
    out[4 * c + 3] = a.w;
  }
}

// C[i][j] = sum_d A[ty + 16 i][d] B[tx + 16 j][d]   (A, B: [64][kLd])
__device__ __forceinline__ void mm_nt(const float* A, const float* B, int ty, int tx, float (&C)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) C[i][j] = 0.f;
#pragma unroll 4
  for (int d = 0; d < kD; ++d) {
    float a[4], bb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A[(ty + 16 * i) * kLd + d];
#pragma unroll
    for (int j = 0; j < 4; ++j) bb[j] = B[(tx + 16 * j) * kLd + d];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) C[i][j] = fmaf(a[i], bb[j], C[i][j]);
  }
}

// C[i][j] += sum_k P[ty + 16 i][k] X[k][tx + 16 j]   (P: [64][kLdP], X: [64][kLd])
__device__ __forceinline__ void mm_nn(const float* Pm, const float* X, int ty, int tx, float (&C)[4][8]) {
#pragma unroll 2
  for (int k = 0; k < kT; ++k) {
    float a[4], bb[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = Pm[(ty + 16 * i) * kLdP + k];
#pragma unroll
    for (int j = 0; j < 8; ++j) bb[j] = X[k * kLd + tx + 16 * j];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) C[i][j] = fmaf(a[i], bb[j], C[i][j]);
  }
}

// C[i][j] += sum_q P[q][ty + 16 i] X[q][tx + 16 j]   (P: [64][kLdP], X: [64][kLd])
__device__ __forceinline__ void mm_tn(const float* Pm, const float* X, int ty, int tx, float (&C)[4][8]) {
#pragma unroll 2
  for (int q = 0; q < kT; ++q) {
    float a[4], bb[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = Pm[q * kLdP + ty + 16 * i];
#pragma unroll
    for (int j = 0; j < 8; ++j) bb[j] = X[q * kLd + tx + 16 * j];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) C[i][j] = fmaf(a[i], bb[j], C[i][j]);
  }
}

// Base-2 score of query i against key j: s * scale * log2(e) plus the mask
// term, -inf where a bool mask is False, beyond the causal diagonal or at
// keys or queries past the sequence ends.
template <int MK, bool CAUSAL>
__device__ __forceinline__ float score2(const Common& c, float s, int b, int h, int i, int j) {
  if (j >= c.Skv || i >= c.Sq) return -INFINITY;
  if (CAUSAL && j > i) return -INFINITY;
  float s2 = s * c.scale_log2;
  if constexpr (MK != kMaskNone) {
    const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j;
    if constexpr (MK == kMaskBool) {
      if (!static_cast<const uint8_t*>(c.mask)[off]) s2 = -INFINITY;
    } else if constexpr (MK == kMaskF32) {
      s2 = fmaf(static_cast<const float*>(c.mask)[off], kLog2e, s2);
    } else {
      s2 = fmaf(__bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]), kLog2e, s2);
    }
  }
  return s2;
}

// Max and sum over the 16 lanes that share ty (lane bits 0-3).
__device__ __forceinline__ float max16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Row transform of a gradient: for row `row` (< nrows) of the raw tensor x
// whose rotated, normed version had gradient g (the thread's 8 columns
// tx + 16 j of the row, the other 120 in the 15 lanes that share ty), writes
//   dx = r g' - (r^3 / D) x (x . g'),  g' = w R^T g
// to out (fp32 row), and returns the row's terms R^T g * x * r of the weight
// gradient in wterm. The rotation partner of column d is d ^ 1, held by lane
// ^ 1. Every lane of the 16 must call it (shuffles).
__device__ __forceinline__ void row_grad(const RowTensor& x, int b, int h, int row, int nrows, const float2* tab,
                                         const float* w, float eps, int tx, const float (&g)[8], float* out,
                                         float (&wterm)[8]) {
  const bool ok = row < nrows;
  const float* xr = static_cast<const float*>(x.p) + b * x.sb + (int64_t)(ok ? row : 0) * x.ss + h * x.sh;
  const float2* t = tab + (int64_t)(ok ? row : 0) * kPairs;
  float xv[8], dy[8], ss = 0.f, xg = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = tx + 16 * j;
    xv[j] = ok ? __ldg(xr + d) : 0.f;
    const float gp = __shfl_xor_sync(0xffffffffu, g[j], 1);  // the partner column's gradient
    const float2 cs = ok ? t[d >> 1] : make_float2(1.f, 0.f);
    // R^T: (g0, g1) -> (g0 cos + g1 sin, g1 cos - g0 sin)
    dy[j] = (d & 1) ? fmaf(g[j], cs.x, -gp * cs.y) : fmaf(g[j], cs.x, gp * cs.y);
    ss = fmaf(xv[j], xv[j], ss);
    xg = fmaf(xv[j], w[d] * dy[j], xg);
  }
  ss = sum16(ss);
  xg = sum16(xg);
  const float rr = rsqrtf(ss * (1.0f / kD) + eps);
  const float c3 = rr * rr * rr * xg * (1.0f / kD);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = tx + 16 * j;
    if (ok) out[d] = fmaf(rr, w[d] * dy[j], -c3 * xv[j]);
    wterm[j] = ok ? dy[j] * xv[j] * rr : 0.f;
  }
}

// The column sums of the block's 64 rows (held as 4 rows per thread, columns
// tx + 16 j) into part[D], in a fixed order: each thread's 4 rows, then the
// 16 row groups (ty) through shared memory.
__device__ __forceinline__ void column_sums(const float (&acc)[4][8], float* red /*[16][D]*/, float* part, int ty,
                                            int tx) {
#pragma unroll
  for (int j = 0; j < 8; ++j) red[ty * kD + tx + 16 * j] = ((acc[0][j] + acc[1][j]) + acc[2][j]) + acc[3][j];
  __syncthreads();
  if (threadIdx.x < kD) {
    float s = 0.f;
    for (int y = 0; y < 16; ++y) s += red[y * kD + threadIdx.x];
    part[threadIdx.x] = s;
  }
}

template <int MK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) f32_fwd_kernel(const __grid_constant__ F32Params P) {
  grid_dependency_wait();
  extern __shared__ float smf[];
  float *sQ = smf, *sK = sQ + kTileF, *sV = sK + kTileF, *sP = sV + kTileF;
  const Common& c = P.c;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, hk = h / c.group;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const float2* tq = c.tab_q + b * c.tab_q_sb;
  const float2* tk = c.tab_k + b * c.tab_k_sb;
  load_rot(sQ, c.q, b, h, qt * kT, c.Sq, tq, c.wq, c.eps);
  float m[4], l[4], O[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) O[i][j] = 0.f;
  }
  int kt_end = tiles64(c.Skv);
  if (CAUSAL) kt_end = min(kt_end, qt + 1);
  for (int kt = 0; kt < kt_end; ++kt) {
    __syncthreads();  // the previous tile's K', V and P are consumed
    load_rot(sK, c.k, b, hk, kt * kT, c.Skv, tk, c.wk, c.eps);
    load_plain(sV, static_cast<const float*>(c.v.p), c.v.sb, c.v.ss, c.v.sh, b, hk, kt * kT, c.Skv);
    __syncthreads();
    float S[4][4];
    mm_nt(sQ, sK, ty, tx, S);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int iq = qt * kT + ty + 16 * i;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        S[i][j] = score2<MK, CAUSAL>(c, S[i][j], b, h, iq, kt * kT + tx + 16 * j);
        mx = fmaxf(mx, S[i][j]);
      }
      const float mn = fmaxf(m[i], max16(mx));
      const float corr = (mn == -INFINITY) ? 1.f : exp2f(m[i] - mn);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = (mn == -INFINITY) ? 0.f : exp2f(S[i][j] - mn);
        rs += p;
        sP[(ty + 16 * i) * kLdP + tx + 16 * j] = p;
      }
      l[i] = l[i] * corr + sum16(rs);
      m[i] = mn;
#pragma unroll
      for (int j = 0; j < 8; ++j) O[i][j] *= corr;
    }
    __syncthreads();
    mm_nn(sP, sV, ty, tx, O);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int iq = qt * kT + ty + 16 * i;
    if (iq >= c.Sq) continue;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
    float* orow = P.o + b * P.o_sb + (int64_t)iq * P.o_ss + h * P.o_sh;
#pragma unroll
    for (int j = 0; j < 8; ++j) orow[tx + 16 * j] = O[i][j] * inv;
    if (tx == 0) P.lse[((int64_t)b * c.H + h) * c.Sq + iq] = l[i] > 0.f ? (m[i] + log2f(l[i])) * kLn2 : -INFINITY;
  }
}

// P and dS of one (query tile, key tile) pair into sP / sdS ([query][key]);
// S = Q' K'^T and dP = dO V^T from the tiles in shared memory.
template <int MK, bool CAUSAL>
__device__ __forceinline__ void p_ds_tile(const F32Params& P, const float* sQ, const float* sK, const float* sdO,
                                          const float* sV, float* sP, float* sdS, int b, int h, int q0, int k0,
                                          int ty, int tx) {
  const Common& c = P.c;
  float S[4][4], dP[4][4];
  mm_nt(sQ, sK, ty, tx, S);
  mm_nt(sdO, sV, ty, tx, dP);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int iq = q0 + ty + 16 * i;
    const bool qok = iq < c.Sq;
    const int64_t ri = ((int64_t)b * c.H + h) * c.Sq + (qok ? iq : 0);
    const float lse = qok ? P.lse_in[ri] : INFINITY;  // -inf (no key) or past S_q: P = 0
    const float l2 = lse == -INFINITY ? INFINITY : lse * kLog2e;
    const float dl = qok ? P.delta[ri] : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float s2 = score2<MK, CAUSAL>(c, S[i][j], b, h, iq, k0 + tx + 16 * j);
      const float p = s2 == -INFINITY ? 0.f : exp2f(s2 - l2);
      sP[(ty + 16 * i) * kLdP + tx + 16 * j] = p;
      sdS[(ty + 16 * i) * kLdP + tx + 16 * j] = p * (dP[i][j] - dl);
    }
  }
}

template <int MK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) f32_bwd_kv_kernel(const __grid_constant__ F32Params P) {
  grid_dependency_wait();
  extern __shared__ float smf[];
  float *sK = smf, *sV = sK + kTileF, *sQ = sV + kTileF, *sdO = sQ + kTileF, *sP = sdO + kTileF, *sdS = sP + kTileP;
  const Common& c = P.c;
  const int kt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const float2* tq = c.tab_q + b * c.tab_q_sb;
  const float2* tk = c.tab_k + b * c.tab_k_sb;
  load_rot(sK, c.k, b, hk, kt * kT, c.Skv, tk, c.wk, c.eps);
  load_plain(sV, static_cast<const float*>(c.v.p), c.v.sb, c.v.ss, c.v.sh, b, hk, kt * kT, c.Skv);
  float dV[4][8], dK[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) dV[i][j] = dK[i][j] = 0.f;
  const int nq = tiles64(c.Sq), q_begin = CAUSAL ? kt : 0;
  for (int g = 0; g < c.group; ++g) {
    const int h = hk * c.group + g;
    for (int qt = q_begin; qt < nq; ++qt) {
      __syncthreads();  // the previous pair's tiles are consumed
      load_rot(sQ, c.q, b, h, qt * kT, c.Sq, tq, c.wq, c.eps);
      load_plain(sdO, P.dout, P.do_sb, P.do_ss, P.do_sh, b, h, qt * kT, c.Sq);
      __syncthreads();
      p_ds_tile<MK, CAUSAL>(P, sQ, sK, sdO, sV, sP, sdS, b, h, qt * kT, kt * kT, ty, tx);
      __syncthreads();
      mm_tn(sP, sdO, ty, tx, dV);
      mm_tn(sdS, sQ, ty, tx, dK);
    }
  }
  // dv; dk from scale dK' (rows = keys ty + 16 i)
  float wt[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = kt * kT + ty + 16 * i;
    float g[8], w8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = dK[i][e] * c.scale;
    float* dkrow = P.dk + b * P.dk_sb + (int64_t)(j < c.Skv ? j : 0) * P.dk_ss + hk * P.dk_sh;
    row_grad(c.k, b, hk, j, c.Skv, tk, c.wk, c.eps, tx, g, dkrow, w8);
#pragma unroll
    for (int e = 0; e < 8; ++e) wt[i][e] = w8[e];
    if (j < c.Skv) {
      float* dvrow = P.dv + b * P.dv_sb + (int64_t)j * P.dv_ss + hk * P.dv_sh;
#pragma unroll
      for (int e = 0; e < 8; ++e) dvrow[tx + 16 * e] = dV[i][e];
    }
  }
  __syncthreads();  // the tiles are free: column sums of the weight-gradient terms
  column_sums(wt, sQ, P.dwk_part + (((int64_t)b * c.Hkv + hk) * gridDim.x + kt) * kD, ty, tx);
}

template <int MK, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) f32_bwd_q_kernel(const __grid_constant__ F32Params P) {
  grid_dependency_wait();
  extern __shared__ float smf[];
  float *sQ = smf, *sdO = sQ + kTileF, *sK = sdO + kTileF, *sV = sK + kTileF, *sdS = sV + kTileF;
  float* sP = sdS;  // P is not kept: only dS feeds dQ'
  const Common& c = P.c;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, hk = h / c.group;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const float2* tq = c.tab_q + b * c.tab_q_sb;
  const float2* tk = c.tab_k + b * c.tab_k_sb;
  load_rot(sQ, c.q, b, h, qt * kT, c.Sq, tq, c.wq, c.eps);
  load_plain(sdO, P.dout, P.do_sb, P.do_ss, P.do_sh, b, h, qt * kT, c.Sq);
  float dQ[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) dQ[i][j] = 0.f;
  int kt_end = tiles64(c.Skv);
  if (CAUSAL) kt_end = min(kt_end, qt + 1);
  for (int kt = 0; kt < kt_end; ++kt) {
    __syncthreads();
    load_rot(sK, c.k, b, hk, kt * kT, c.Skv, tk, c.wk, c.eps);
    load_plain(sV, static_cast<const float*>(c.v.p), c.v.sb, c.v.ss, c.v.sh, b, hk, kt * kT, c.Skv);
    __syncthreads();
    p_ds_tile<MK, CAUSAL>(P, sQ, sK, sdO, sV, sP, sdS, b, h, qt * kT, kt * kT, ty, tx);
    __syncthreads();
    mm_nn(sdS, sK, ty, tx, dQ);
  }
  float wt[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int iq = qt * kT + ty + 16 * i;
    float g[8], w8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = dQ[i][e] * c.scale;
    float* dqrow = P.dq + b * P.dq_sb + (int64_t)(iq < c.Sq ? iq : 0) * P.dq_ss + h * P.dq_sh;
    row_grad(c.q, b, h, iq, c.Sq, tq, c.wq, c.eps, tx, g, dqrow, w8);
#pragma unroll
    for (int e = 0; e < 8; ++e) wt[i][e] = w8[e];
  }
  __syncthreads();
  column_sums(wt, sQ, P.dwq_part + (((int64_t)b * c.H + h) * gridDim.x + qt) * kD, ty, tx);
}

template <class K>
cudaError_t launch_f32(K kern, dim3 grid, uint32_t smem, std::atomic<uint64_t>& done, const F32Params& p,
                       cudaStream_t stream) {
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  return launch_chained(kern, grid, dim3(kThreads), smem, stream, p);
}

template <int MK, bool CAUSAL>
cudaError_t f32_fwd_t(const F32Params& p, cudaStream_t stream) {
  static std::atomic<uint64_t> done{0};
  return launch_f32(f32_fwd_kernel<MK, CAUSAL>, dim3((p.c.Sq + kT - 1) / kT, p.c.H, p.c.B), kFwdSmemF, done, p,
                    stream);
}

template <int MK, bool CAUSAL>
cudaError_t f32_bwd_kv_t(const F32Params& p, cudaStream_t stream) {
  static std::atomic<uint64_t> done{0};
  return launch_f32(f32_bwd_kv_kernel<MK, CAUSAL>, dim3((p.c.Skv + kT - 1) / kT, p.c.Hkv, p.c.B), kBwdKVSmemF, done, p,
                    stream);
}

template <int MK, bool CAUSAL>
cudaError_t f32_bwd_q_t(const F32Params& p, cudaStream_t stream) {
  static std::atomic<uint64_t> done{0};
  return launch_f32(f32_bwd_q_kernel<MK, CAUSAL>, dim3((p.c.Sq + kT - 1) / kT, p.c.H, p.c.B), kBwdQSmemF, done, p,
                    stream);
}

}  // namespace

cudaError_t launch_f32_fwd(const F32Params& p, cudaStream_t stream) {
  if (p.c.causal) return f32_fwd_t<kMaskNone, true>(p, stream);
  switch (p.c.mask_kind) {
    case kMaskBool: return f32_fwd_t<kMaskBool, false>(p, stream);
    case kMaskF32: return f32_fwd_t<kMaskF32, false>(p, stream);
    case kMaskBF16: return f32_fwd_t<kMaskBF16, false>(p, stream);
    default: return f32_fwd_t<kMaskNone, false>(p, stream);
  }
}

cudaError_t launch_f32_bwd_kv(const F32Params& p, cudaStream_t stream) {
  if (p.c.causal) return f32_bwd_kv_t<kMaskNone, true>(p, stream);
  switch (p.c.mask_kind) {
    case kMaskBool: return f32_bwd_kv_t<kMaskBool, false>(p, stream);
    case kMaskF32: return f32_bwd_kv_t<kMaskF32, false>(p, stream);
    case kMaskBF16: return f32_bwd_kv_t<kMaskBF16, false>(p, stream);
    default: return f32_bwd_kv_t<kMaskNone, false>(p, stream);
  }
}

cudaError_t launch_f32_bwd_q(const F32Params& p, cudaStream_t stream) {
  if (p.c.causal) return f32_bwd_q_t<kMaskNone, true>(p, stream);
  switch (p.c.mask_kind) {
    case kMaskBool: return f32_bwd_q_t<kMaskBool, false>(p, stream);
    case kMaskF32: return f32_bwd_q_t<kMaskF32, false>(p, stream);
    case kMaskBF16: return f32_bwd_q_t<kMaskBF16, false>(p, stream);
    default: return f32_bwd_q_t<kMaskNone, false>(p, stream);
  }
}

}  // namespace st
