// Small kernels around the two attention kernels:
//  - rotary table:   position ids -> (cos, sin) per token and pair (fp32);
//  - mask classify:  bool mask tiles -> {all True, all False, mixed}, plus the
//                    "whole mask is all True" counter;
//  - backward pre:   Delta_i = sum_d dO_id O_id, zero the fp32 dQ accumulator;
//  - dq post:        fp32 gradient rows of the rotated, normed q (or k) ->
//                    inverse rotation -> RMSNorm backward -> dq (or dk), with
//                    per-block partial sums of the norm-weight gradient;
//  - dw reduce:      fixed-order sums of the weight-gradient partials.
#include "st_aux.h"

namespace st {

namespace {

// (b, i, h) of row `row` of a [B, S, H] row space; 32-bit arithmetic when the
// row count allows it (a 64-bit division is a long software sequence).
struct RowIdx {
  int b, i, h;
};
__device__ __forceinline__ RowIdx row_idx(int64_t row, int S, int H, bool small) {
  RowIdx r;
  if (small) {
    const uint32_t rw = static_cast<uint32_t>(row), t = rw / static_cast<uint32_t>(H);
    r.h = static_cast<int>(rw - t * static_cast<uint32_t>(H));
    r.b = static_cast<int>(t / static_cast<uint32_t>(S));
    r.i = static_cast<int>(t - static_cast<uint32_t>(r.b) * static_cast<uint32_t>(S));
  } else {
    const int64_t t = row / H;
    r.h = static_cast<int>(row - t * H);
    r.b = static_cast<int>(t / S);
    r.i = static_cast<int>(t - static_cast<int64_t>(r.b) * S);
  }
  return r;
}

static_assert(kPairs == 64, "the table kernel indexes pairs with shifts");

// Element e of a caller table as fp32.
__device__ __forceinline__ float table_elem(const void* t, int dtype, int64_t e) {
  if (dtype == kTabF32) return static_cast<const float*>(t)[e];
  if (dtype == kTabBF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(t)[e]);
  return __half2float(static_cast<const __half*>(t)[e]);
}

// (cos, sin) of id * omega_p, the angle reduced to [-pi, pi] in fp64 before
// the fp32 sincosf so that large ids keep full fp32 accuracy; or, in the table
// form, entry 2p of the caller's pair-duplicated cos/sin rows.
__global__ void table_kernel(const __grid_constant__ TableParams p) {
  grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x < kCtrlWords && p.ctrl) p.ctrl[threadIdx.x] = 0u;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.n_zero; e += (int64_t)gridDim.x * blockDim.x)
    p.zero[e] = 0u;
  const int64_t n = (int64_t)p.Bt * p.S * kPairs;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int pr = static_cast<int>(e & (kPairs - 1));
    const int64_t tok = e >> 6;  // kPairs = 64
    const int bt = p.Bt == 1 ? 0 : static_cast<int>(tok / p.S);
    const int s = static_cast<int>(tok - static_cast<int64_t>(bt) * p.S);
    if (p.cos) {
      const float cs = table_elem(p.cos, p.tab_dtype, bt * p.c_sb + (int64_t)s * p.c_ss + (int64_t)(2 * pr) * p.c_sd);
      const float sn = table_elem(p.sin, p.tab_dtype, bt * p.s_sb + (int64_t)s * p.s_ss + (int64_t)(2 * pr) * p.s_sd);
      p.out[e] = make_float2(cs, sn);
      p.out16[e] = __floats2half2_rn(cs, sn);
      continue;
    }
    const int a = p.axis_of[pr];
    const int64_t off = bt * p.i_sb + (int64_t)s * p.i_ss + (int64_t)a * p.i_sa;
    const double id = p.ids_f32 ? static_cast<double>(static_cast<const float*>(p.ids)[off])
                                : static_cast<double>(static_cast<const int32_t*>(p.ids)[off]);
    const double phi = id * p.omega[pr];
    const double k = rint(phi * 0.15915494309189535);  // 1 / (2 pi)
    const double red = fma(-k, 6.283185307179586, phi);
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    p.out[e] = make_float2(cs, sn);
    p.out16[e] = __floats2half2_rn(cs, sn);
  }
}

__global__ void classify_kernel(const __grid_constant__ ClassifyParams p) {
  grid_dependency_wait();
  const int kt = blockIdx.x, qt = blockIdx.y;
  const int bm = blockIdx.z / p.Hm, hm = blockIdx.z % p.Hm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = (p.Sqm == 1) ? 1 : min(kTile, p.Sqm - qt * kTile);
  const int keys = min(kTile, p.Skv - kt * kTile);
  bool any_t = false, any_f = false;
  for (int r = warp; r < rows; r += blockDim.x / 32) {
    const uint8_t* row = p.mask + bm * p.m_sb + hm * p.m_sh + (int64_t)(qt * kTile + r) * p.m_sq + kt * kTile;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = 4 * lane + u;
      if (jj < keys) {
        if (__ldg(row + jj)) any_t = true; else any_f = true;
      }
    }
  }
  const int bt = __syncthreads_or(any_t);
  const int bf = __syncthreads_or(any_f);
  __shared__ int is_last;
  if (threadIdx.x == 0) {
    const uint8_t flag = !bf ? kTileAllTrue : (!bt ? kTileAllFalse : kTileMixed);
    p.flags[((int64_t)blockIdx.z * p.nQtm + qt) * p.nKt + kt] = flag;
    if (bf) atomicOr(p.ctrl + kCtrlAnyFalse, 1u);
    __threadfence();
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    is_last = (atomicAdd(p.ctrl + kCtrlClassifyDone, 1u) == total - 1);
  }
  __syncthreads();
  if (is_last && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.ctrl + kCtrlAnyFalse, 0u) == 0u) atomicAdd(p.counters + kCtrMaskAllTrue, 1ull);
  }
}

// kPreRows (b, i, h) rows per warp, their loads issued together; lane l
// owns head dims 4l..4l+3 of each row. Block 0 also clears the weight-gradient
// reduction counters (the table kernel, which clears them otherwise, may be
// skipped by a backward that reuses the forward's tables).
constexpr int kPreRows = 2;

__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ PreParams p) {
  grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x < 2 && p.ctrl) p.ctrl[kCtrlDwDone + threadIdx.x] = 0u;
  const int lane = threadIdx.x & 31;
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const bool small = nrows < (int64_t(1) << 31);
  const int64_t row0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kPreRows;
  // lane u < kPreRows splits row row0 + u into (b, i, h) once; the warp reads
  // it by shuffles (the divisions cost more than the row's loads otherwise)
  RowIdx mine = {0, 0, 0};
  if (lane < kPreRows && row0 + lane < nrows) mine = row_idx(row0 + lane, p.Sq, p.H, small);
  float o[kPreRows][4], g[kPreRows][4];
#pragma unroll
  for (int u = 0; u < kPreRows; ++u) {
    const int64_t row = row0 + u;
    const int b = __shfl_sync(0xffffffffu, mine.b, u), i = __shfl_sync(0xffffffffu, mine.i, u),
              h = __shfl_sync(0xffffffffu, mine.h, u);
    if (row >= nrows) {
#pragma unroll
      for (int e = 0; e < 4; ++e) o[u][e] = g[u][e] = 0.f;
      continue;
    }
    const int64_t oo = b * p.o_sb + (int64_t)i * p.o_ss + h * p.o_sh + 4 * lane;
    const int64_t go = b * p.do_sb + (int64_t)i * p.do_ss + h * p.do_sh + 4 * lane;
    if (p.o_dt == kDtF32) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.o) + oo));
      const float4 w = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.dout) + go));
      o[u][0] = v.x; o[u][1] = v.y; o[u][2] = v.z; o[u][3] = v.w;
      g[u][0] = w.x; g[u][1] = w.y; g[u][2] = w.z; g[u][3] = w.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.o) + oo));
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.dout) + go));
      const bool h = p.o_dt == kDtF16;
      o[u][0] = h ? f16_lo(v.x) : bf16_lo(v.x); o[u][1] = h ? f16_hi(v.x) : bf16_hi(v.x);
      o[u][2] = h ? f16_lo(v.y) : bf16_lo(v.y); o[u][3] = h ? f16_hi(v.y) : bf16_hi(v.y);
      g[u][0] = h ? f16_lo(w.x) : bf16_lo(w.x); g[u][1] = h ? f16_hi(w.x) : bf16_hi(w.x);
      g[u][2] = h ? f16_lo(w.y) : bf16_lo(w.y); g[u][3] = h ? f16_hi(w.y) : bf16_hi(w.y);
    }
  }
#pragma unroll
  for (int u = 0; u < kPreRows; ++u) {
    const int64_t row = row0 + u;
    if (row < nrows && p.dq_acc) reinterpret_cast<float4*>(p.dq_acc + row * kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float acc[kPreRows];
#pragma unroll
  for (int u = 0; u < kPreRows; ++u) acc[u] = o[u][0] * g[u][0] + o[u][1] * g[u][1] + o[u][2] * g[u][2] + o[u][3] * g[u][3];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int u = 0; u < kPreRows; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
  }
  if (lane < kPreRows) {
    float a = acc[0];
#pragma unroll
    for (int u = 1; u < kPreRows; ++u)
      if (lane == u) a = acc[u];
    if (row0 + lane < nrows) p.delta[((int64_t)mine.b * p.H + mine.h) * p.Sq + mine.i] = a;
  }
}

// One warp per (b, i, h) row, 128 rows per block (8 warps x 16 rows). Lane l
// owns head dims 4l..4l+3 (rotation pairs 2l, 2l+1), so every row load and
// store is one coalesced access per warp; the row's sums (x.x, x.g) are warp
// shuffles. With dy = R^T g (sin negated) and g' = w dy:
//   dx = r g' - (r^3 / D) x (x . g'); the weight gradient gathers dy x r.
constexpr int kPostWarps = 8;
constexpr int kPostThreads = kPostWarps * 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kPostRows = 1;  // rows per warp and pass, their loads issued together

__global__ void __launch_bounds__(kPostThreads) dq_post_kernel(const __grid_constant__ PostParams p) {
  grid_dependency_wait();
  __shared__ float4 part[kPostWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const bool small = nrows < (int64_t(1) << 31);
  const int64_t row0 = (int64_t)blockIdx.x * kPostBlockRows;
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.wq) + lane);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
  for (int k0 = warp * kPostRows; k0 < kPostBlockRows; k0 += kPostWarps * kPostRows) {
    float4 g[kPostRows], x[kPostRows], cs[kPostRows];
    int64_t yoff[kPostRows];
    bool valid[kPostRows];
#pragma unroll
    for (int u = 0; u < kPostRows; ++u) {
      const int64_t row = row0 + k0 + u;
      valid[u] = row < nrows;
      const int64_t rr = valid[u] ? row : 0;
      const RowIdx x3 = row_idx(rr, p.Sq, p.H, small);
      const int b = x3.b, i = x3.i, h = x3.h;
      g[u] = __ldg(reinterpret_cast<const float4*>(p.dq_acc + rr * kD) + lane);
      const int64_t xoff = b * p.q.sb + (int64_t)i * p.q.ss + h * p.q.sh + 4 * lane;
      if (p.q.dt == kDtF32) {
        x[u] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.q.p) + xoff));
      } else {
        const uint2 t = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q.p) + xoff));
        x[u] = p.q.dt == kDtF16 ? make_float4(f16_lo(t.x), f16_hi(t.x), f16_lo(t.y), f16_hi(t.y))
                                : make_float4(bf16_lo(t.x), bf16_hi(t.x), bf16_lo(t.y), bf16_hi(t.y));
      }
      cs[u] = __ldg(reinterpret_cast<const float4*>(p.tab_q + b * p.tab_q_sb + (int64_t)i * kPairs) + lane);
      yoff[u] = b * p.dq_sb + (int64_t)i * p.dq_ss + h * p.dq_sh + 4 * lane;
    }
    float ss[kPostRows];
#pragma unroll
    for (int u = 0; u < kPostRows; ++u)
      ss[u] = x[u].x * x[u].x + x[u].y * x[u].y + x[u].z * x[u].z + x[u].w * x[u].w;
    // inverse rotation of the two pairs: (cos, sin) = (cs.x, cs.y), (cs.z, cs.w)
    float4 gw[kPostRows];
    float xg[kPostRows];
#pragma unroll
    for (int u = 0; u < kPostRows; ++u) {
      const float4 gg = g[u], c4 = cs[u];
      const float d0 = gg.x * c4.x + gg.y * c4.y, d1 = -gg.x * c4.y + gg.y * c4.x;
      const float d2 = gg.z * c4.z + gg.w * c4.w, d3 = -gg.z * c4.w + gg.w * c4.z;
      g[u] = make_float4(d0, d1, d2, d3);  // dy
      gw[u] = make_float4(w.x * d0, w.y * d1, w.z * d2, w.w * d3);
      xg[u] = x[u].x * gw[u].x + x[u].y * gw[u].y + x[u].z * gw[u].z + x[u].w * gw[u].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int u = 0; u < kPostRows; ++u) {
        ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
        xg[u] += __shfl_xor_sync(0xffffffffu, xg[u], o);
      }
    }
#pragma unroll
    for (int u = 0; u < kPostRows; ++u) {
      if (!valid[u]) continue;
      const float r = rsqrtf(ss[u] * (1.0f / kD) + p.eps);
      const float4 xx = x[u], dy = g[u], q = gw[u];
      acc.x = fmaf(dy.x, xx.x * r, acc.x);
      acc.y = fmaf(dy.y, xx.y * r, acc.y);
      acc.z = fmaf(dy.z, xx.z * r, acc.z);
      acc.w = fmaf(dy.w, xx.w * r, acc.w);
      const float c3 = r * r * r * xg[u] * (1.0f / kD);
      const float y0 = r * q.x - c3 * xx.x, y1 = r * q.y - c3 * xx.y, y2 = r * q.z - c3 * xx.z, y3 = r * q.w - c3 * xx.w;
      if (p.dq_dt == kDtF32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.dq) + yoff[u]) = make_float4(y0, y1, y2, y3);
      } else {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.dq) + yoff[u]) =
            make_uint2(pack_dt(p.dq_dt, y0, y1), pack_dt(p.dq_dt, y2, y3));
      }
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (threadIdx.x < kD) {  // column d = 4 * lane + component, summed over the warps in order
    const int l = threadIdx.x >> 2, comp = threadIdx.x & 3;
    float sum = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < kPostWarps; ++w8) {
      const float4 v = part[w8][l];
      sum += comp == 0 ? v.x : comp == 1 ? v.y : comp == 2 ? v.z : v.w;
    }
    p.dwq_part[(int64_t)blockIdx.x * kD + threadIdx.x] = sum;
  }
}

// Grid (nblocks, 2): y = 0 reduces the q-weight partials, y = 1 the k-weight
// partials. Each block sums up to kDwChunk partials in index order; the last
// block to finish sums the block results in index order.
__global__ void __launch_bounds__(128) dw_reduce_kernel(const __grid_constant__ DwParams p) {
  grid_dependency_wait();
  const int which = blockIdx.y, tid = threadIdx.x;
  const float* part = which ? p.dwk_part : p.dwq_part;
  const int n = which ? p.n_k : p.n_q;
  float* scratch = p.scratch + (int64_t)which * gridDim.x * kD;
  const int p0 = blockIdx.x * kDwChunk;
  const int p1 = min(n, p0 + kDwChunk);
  float acc = 0.f;
  int q = p0;
  for (; q + 8 <= p1; q += 8) {  // loads of eight partials in flight, added in index order
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + (int64_t)(q + u) * kD + tid);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc += v[u];
  }
  for (; q < p1; ++q) acc += __ldcg(part + (int64_t)q * kD + tid);
  scratch[(int64_t)blockIdx.x * kD + tid] = acc;
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (tid == 0) is_last = (atomicAdd(p.ctrl + kCtrlDwDone + which, 1u) == gridDim.x - 1);
  __syncthreads();
  if (is_last) {
    __threadfence();
    float tot = 0.f;
    for (int b = 0; b < (int)gridDim.x; ++b) tot += __ldcg(scratch + (int64_t)b * kD + tid);
    (which ? p.dwk : p.dwq)[tid] = tot;
  }
}

// Self-test of the bounded waits: one thread waits on an mbarrier that nothing
// ever arrives on, gives up after `budget` clock64 cycles and records the
// timeout exactly as the attention kernels do.
__global__ void wait_probe_kernel(unsigned* status, unsigned long long* counters, long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, budget)) {
      atomicOr(status, kStatusTimeout);
      atomicAdd(counters + kCtrTimeouts, 1ull);
    }
  }
}

}  // namespace

cudaError_t launch_wait_probe(unsigned* status, unsigned long long* counters, long long budget, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status, counters, budget);
  return cudaGetLastError();
}

cudaError_t launch_table(const TableParams& p, cudaStream_t stream) {
  const int64_t n = (int64_t)p.Bt * p.S * kPairs;
  const int threads = 256;
  int blocks = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 152 * 16));
  if (blocks < 1) blocks = 1;
  return launch_chained(table_kernel, dim3(blocks), dim3(threads), 0, stream, p);
}

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t stream) {
  dim3 grid(p.nKt, p.nQtm, p.Bm * p.Hm);
  return launch_chained(classify_kernel, grid, dim3(128), 0, stream, p);
}

cudaError_t launch_bwd_pre(const PreParams& p, cudaStream_t stream) {
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const int64_t warps = (nrows + kPreRows - 1) / kPreRows;
  const int64_t blocks = (warps * 32 + 255) / 256;
  return launch_chained(bwd_pre_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

cudaError_t launch_dq_post(const PostParams& p, cudaStream_t stream) {
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const int64_t blocks = (nrows + kPostBlockRows - 1) / kPostBlockRows;
  return launch_chained(dq_post_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPostThreads), 0, stream, p);
}

// One thread per row, with the forward prologues' arithmetic in their order,
// so that the rows equal the ones a forward leaves in the workspace:
// r = 1/sqrt(mean x^2 + eps) (16-bit q: the sum of squares of each 64-dim half
// with separate even/odd accumulators, as the two lanes of a row do; fp32 q:
// the in-order sums of the four 32-dim quarters added as ((s0 + s1) + (s2 +
// s3)), as the four lanes of a row do), n = x w r,
// y = (n0 cos - n1 sin, n0 sin + n1 cos) with the fp16 (16-bit q) or fp32
// (fp32 q) table, rounded once to the operand type.
__global__ void __launch_bounds__(128) qprime_kernel(const __grid_constant__ QPrimeParams p) {
  grid_dependency_wait();
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= nrows) return;
  const RowIdx x = row_idx(row, p.Sq, p.H, nrows < (int64_t(1) << 31));
  const int64_t off = x.b * p.q.sb + (int64_t)x.i * p.q.ss + x.h * p.q.sh;
  const int64_t trow = x.b * p.tab_sb + (int64_t)x.i * kPairs;
  uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * kD);
  const float4* w4 = reinterpret_cast<const float4*>(p.w);
  if (p.q.dt != kDtF32) {
    const bool f16 = p.q.dt == kDtF16;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q.p) + off);
    float half_ss[2];
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = __ldg(src + 8 * hh + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = f16 ? f16_lo(u[e]) : bf16_lo(u[e]), hi = f16 ? f16_hi(u[e]) : bf16_hi(u[e]);
          a0 = fmaf(lo, lo, a0);
          a1 = fmaf(hi, hi, a1);
        }
      }
      half_ss[hh] = a0 + a1;
    }
    const float r = rsqrtf((half_ss[0] + half_ss[1]) * (1.0f / kD) + p.eps);
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {  // dims 8c .. 8c + 7
      const uint4 v = __ldg(src + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      const float4 wa = __ldg(w4 + 2 * c), wb = __ldg(w4 + 2 * c + 1);
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 sc = __half22float2(p.tab16[trow + 4 * c + e]);
        const float lo = f16 ? f16_lo(u[e]) : bf16_lo(u[e]), hi = f16 ? f16_hi(u[e]) : bf16_hi(u[e]);
        const float n0 = lo * wv[2 * e] * r, n1 = hi * wv[2 * e + 1] * r;
        const float y0 = n0 * sc.x - n1 * sc.y, y1 = n0 * sc.y + n1 * sc.x;
        o4[e] = p.f16 ? pack16<true>(y0, y1) : pack16<false>(y0, y1);
      }
      out[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.q.p) + off);
    float sq[4];  // sums of squares of the four 32-dim quarters, each in order
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      float s4 = 0.f;
#pragma unroll
      for (int c = 8 * k4; c < 8 * k4 + 8; ++c) {
        const float4 v = __ldg(src + c);
        s4 = fmaf(v.x, v.x, s4);
        s4 = fmaf(v.y, v.y, s4);
        s4 = fmaf(v.z, v.z, s4);
        s4 = fmaf(v.w, v.w, s4);
      }
      sq[k4] = s4;
    }
    const float r = rsqrtf(((sq[0] + sq[1]) + (sq[2] + sq[3])) * (1.0f / kD) + p.eps);
    const float4* t4 = reinterpret_cast<const float4*>(p.tab + trow);
#pragma unroll 1
    for (int c = 0; c < kD / 8; ++c) {
      uint32_t o4[4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float4 v = __ldg(src + 2 * c + hh);
        const float4 cs = __ldg(t4 + 2 * c + hh);
        const float4 ww = __ldg(w4 + 2 * c + hh);
        const float n0 = v.x * ww.x * r, n1 = v.y * ww.y * r, n2 = v.z * ww.z * r, n3 = v.w * ww.w * r;
        const float y0 = n0 * cs.x - n1 * cs.y, y1 = n0 * cs.y + n1 * cs.x;
        const float y2 = n2 * cs.z - n3 * cs.w, y3 = n2 * cs.w + n3 * cs.z;
        o4[2 * hh] = p.f16 ? pack16<true>(y0, y1) : pack16<false>(y0, y1);
        o4[2 * hh + 1] = p.f16 ? pack16<true>(y2, y3) : pack16<false>(y2, y3);
      }
      out[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
}

cudaError_t launch_qprime(const QPrimeParams& p, cudaStream_t stream) {
  const int64_t nrows = (int64_t)p.B * p.Sq * p.H;
  const int64_t blocks = (nrows + 127) / 128;
  return launch_chained(qprime_kernel, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, stream, p);
}

cudaError_t launch_dw_reduce(const DwParams& p, cudaStream_t stream) {
  dim3 grid(dw_reduce_blocks(p.n_q, p.n_k), 2);
  return launch_chained(dw_reduce_kernel, grid, dim3(kD), 0, stream, p);
}

}  // namespace st
