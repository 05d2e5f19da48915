// C-ABI host layer: argument validation, workspace planning, kernel launches
// and the dispatch counters. Nothing here allocates device memory or
// synchronises a stream, except st_get_stats and st_check_status.
#include <atomic>
#include <mutex>
#include <vector>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include <cudaTypedefs.h>

#include "st_rope_attn.h"
#include "st_aux.h"
#include "st_f32.h"
#include "st_kernels.h"

namespace st {
__device__ unsigned g_status = 0;
__device__ unsigned long long g_counters[kNumCounters];
}  // namespace st

namespace {

using namespace st;

thread_local std::string t_err;
std::atomic<uint64_t> h_fwd_calls{0}, h_bwd_calls{0}, h_mixed{0}, h_launches{0};

// ---- optional per-kernel event timing (measurement only)
struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_tmu;
std::atomic<bool> g_timing{false};
std::vector<TimedLaunch> g_pending;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launches one kernel through `fn`, counting it and, when timing is on,
// bracketing it with events on its stream.
template <class F>
cudaError_t launch_counted(int kind, cudaStream_t stream, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (g_timing.load(std::memory_order_relaxed)) {
    std::lock_guard<std::mutex> lk(g_tmu);
    a = take_event();
    b = take_event();
    if (a) cudaEventRecord(a, stream);
  }
  cudaError_t e = fn();
  if (e == cudaSuccess) ++h_launches;
  if (a && b) {
    cudaEventRecord(b, stream);
    std::lock_guard<std::mutex> lk(g_tmu);
    g_pending.push_back({kind, a, b});
  }
  return e;
}

st_status fail(st_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

int elem_bytes(int dt) {
  switch (dt) {
    case ST_BF16: case ST_F16: return 2;
    case ST_F32: case ST_I32: return 4;
    case ST_BOOL: return 1;
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long wait_budget() {
  static long long v = [] {
    const char* e = std::getenv("ST_WAIT_BUDGET");
    long long b = e ? std::atoll(e) : 0;
    return b > 0 ? b : (1ll << 31);  // ~1 s of clock64 at GB300 clocks
  }();
  return v;
}

struct Dev {
  unsigned* status = nullptr;
  unsigned long long* counters = nullptr;
};

st_status device_globals(Dev* d) {
  static Dev cache[64];
  static std::atomic<bool> ready[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(ST_ERR_CUDA, "cudaGetDevice failed");
  if (!ready[dev].load(std::memory_order_acquire)) {
    Dev v;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&v.status), g_status) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&v.counters), g_counters) != cudaSuccess)
      return fail(ST_ERR_CUDA, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(cudaGetLastError()));
    cache[dev] = v;
    ready[dev].store(true, std::memory_order_release);
  }
  *d = cache[dev];
  return ST_OK;
}

// ------------------------------------------------------------- validation
struct Shape {
  int B = 0, Sq = 0, Skv = 0, H = 0, D = 0;
  int Hkv = 0;  // K/V heads: H is a multiple of it (grouped K/V heads)
};

static_assert(kDtBF16 == ST_BF16 && kDtF16 == ST_F16 && kDtF32 == ST_F32, "row dtype codes");

constexpr unsigned bit(int dt) { return 1u << dt; }

// A [B, S, H, D] tensor whose dtype is one of `dts` (a set of bit(st_dtype)).
st_status check_bshd(const st_tensor* t, const char* name, int B, int S, int H, int D, unsigned dts,
                     RowTensor* out) {
  if (!t) return fail(ST_ERR_INVALID_ARG, "%s is NULL", name);
  if (t->ndim != 4) return fail(ST_ERR_SHAPE, "%s must be 4-D [B,S,H,D], got ndim=%d", name, t->ndim);
  if (t->shape[0] != B || t->shape[1] != S || t->shape[2] != H || t->shape[3] != D)
    return fail(ST_ERR_SHAPE, "%s has shape [%lld,%lld,%lld,%lld], expected [%d,%d,%d,%d]", name,
                (long long)t->shape[0], (long long)t->shape[1], (long long)t->shape[2], (long long)t->shape[3], B,
                S, H, D);
  if (t->dtype < 0 || t->dtype > 31 || !(dts & bit(t->dtype)))
    return fail(ST_ERR_DTYPE, "%s has unsupported dtype %d", name, t->dtype);
  const int64_t n = (int64_t)B * S * H;
  if (n > 0) {
    if (!t->data) return fail(ST_ERR_INVALID_ARG, "%s data is NULL", name);
    const int eb = elem_bytes(t->dtype);
    if (t->stride[3] != 1) return fail(ST_ERR_ALIGN, "%s must have unit stride on D", name);
    if (!aligned16(t->data)) return fail(ST_ERR_ALIGN, "%s data pointer is not 16-byte aligned", name);
    for (int a = 0; a < 3; ++a)
      if (t->shape[a] > 1 && ((t->stride[a] * eb) % 16) != 0)
        return fail(ST_ERR_ALIGN, "%s stride[%d]=%lld elements is not a multiple of 16 bytes", name, a,
                    (long long)t->stride[a]);
  }
  if (out) {
    out->p = t->data;
    out->sb = t->shape[0] > 1 ? t->stride[0] : 0;
    out->ss = t->shape[1] > 1 ? t->stride[1] : 0;
    out->sh = t->shape[2] > 1 ? t->stride[2] : 0;
    out->dt = t->dtype;
  }
  return ST_OK;
}

st_status check_vec(const st_tensor* t, const char* name, int D) {
  if (!t || !t->data) return fail(ST_ERR_INVALID_ARG, "%s is NULL", name);
  if (t->ndim != 1 || t->shape[0] != D) return fail(ST_ERR_SHAPE, "%s must be [%d]", name, D);
  if (t->dtype != ST_F32) return fail(ST_ERR_DTYPE, "%s must be fp32", name);
  if (t->stride[0] != 1) return fail(ST_ERR_ALIGN, "%s must be contiguous", name);
  if (!aligned16(t->data)) return fail(ST_ERR_ALIGN, "%s data pointer is not 16-byte aligned", name);
  return ST_OK;
}

// The rotation source of q or of k: position ids (t), or in the table form
// the caller's cos (t) and sin tables.
struct Ids {
  const st_tensor* t;
  int Bt, S;
  const st_tensor* sin = nullptr;
  bool table = false;
};

st_status check_ids(const st_tensor* t, const char* name, int B, int S, int n_axes, Ids* out) {
  if (!t || (!t->data && S > 0)) return fail(ST_ERR_INVALID_ARG, "%s is NULL", name);
  if (t->ndim != 3) return fail(ST_ERR_SHAPE, "%s must be 3-D [B|1, S, n_axes]", name);
  if (!(t->shape[0] == 1 || t->shape[0] == B) || t->shape[1] != S || t->shape[2] != n_axes)
    return fail(ST_ERR_SHAPE, "%s has shape [%lld,%lld,%lld], expected [%d|1,%d,%d]", name, (long long)t->shape[0],
                (long long)t->shape[1], (long long)t->shape[2], B, S, n_axes);
  if (t->dtype != ST_I32 && t->dtype != ST_F32) return fail(ST_ERR_DTYPE, "%s must be int32 or fp32", name);
  out->t = t;
  out->Bt = static_cast<int>(t->shape[0]);
  out->S = S;
  return ST_OK;
}

static_assert(kTabBF16 == ST_BF16 && kTabF16 == ST_F16 && kTabF32 == ST_F32, "table dtype codes");

// The pages' table form: pair-duplicated cos/sin of shape [S, D], [1, S, D]
// or [B, S, D], fp32, bf16 or fp16 (the same for both), any element strides.
st_status check_tables(const st_tensor* c, const st_tensor* sn, const char* name, int B, int S, Ids* out) {
  if (!c || !sn) return fail(ST_ERR_INVALID_ARG, "%s: cos and sin must both be given", name);
  if (c->ndim != sn->ndim || (c->ndim != 2 && c->ndim != 3))
    return fail(ST_ERR_SHAPE, "%s must both be [S, D] or [B|1, S, D]", name);
  const int o = c->ndim - 2;
  const int64_t bt = c->ndim == 3 ? c->shape[0] : 1;
  for (const st_tensor* t : {c, sn}) {
    if ((c->ndim == 3 && t->shape[0] != bt) || t->shape[o] != S || t->shape[o + 1] != kD)
      return fail(ST_ERR_SHAPE, "%s must have shape [%d, %d] or [%d|1, %d, %d]", name, S, kD, B, S, kD);
  }
  if (!(bt == 1 || bt == B)) return fail(ST_ERR_SHAPE, "%s batch dim is %lld, expected 1 or %d", name, (long long)bt, B);
  if (c->dtype != sn->dtype) return fail(ST_ERR_DTYPE, "%s must have the same dtype", name);
  if (c->dtype != ST_F32 && c->dtype != ST_BF16 && c->dtype != ST_F16)
    return fail(ST_ERR_DTYPE, "%s must be fp32, bf16 or fp16", name);
  if ((!c->data || !sn->data) && bt * S > 0) return fail(ST_ERR_INVALID_ARG, "%s data is NULL", name);
  out->t = c;
  out->sin = sn;
  out->table = true;
  out->Bt = static_cast<int>(bt);
  out->S = S;
  return ST_OK;
}

struct Plan {
  Shape sh;
  RowTensor q, k, v;
  Ids ids_q{}, ids_k{};
  bool separate_k_table = false;
  int mask_kind = kMaskNone;
  int Bm = 1, Hm = 1, Sqm = 1;
  int64_t m_sb = 0, m_sh = 0, m_sq = 0;
  int nQt = 0, nKt = 0, nQtm = 1;
  // workspace offsets
  size_t off_tab16_q = 0, off_tab16_k = 0;
  size_t off_ctrl = 0, off_tab_q = 0, off_tab_k = 0, off_flags = 0, off_delta = 0, off_dqacc = 0,
         off_dwk = 0, off_dwq = 0, off_dwscratch = 0, off_qp = 0, total = 0;
  size_t off_kflags = 0, off_kcache = 0;
  size_t fwd_base = 0;  // the forward's bytes without the K' tile cache
  bool kcache = false;  // the forward part ends with the K' tile cache
  int n_dwq = 0, n_dwk = 0;
  bool f32 = false;  // q, k, v all fp32: the exact-fp32 kernels
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

st_status plan_call(const st_tensor* q, const st_tensor* k, const st_tensor* v, const st_tensor* mask, int causal,
                    const st_rope* rope, int for_backward, Plan* P) {
  if (!q || !k || !v) return fail(ST_ERR_INVALID_ARG, "q, k and v must not be NULL");
  if (q->ndim != 4 || k->ndim != 4) return fail(ST_ERR_SHAPE, "q and k must be 4-D [B,S,H,D]");
  Shape s;
  s.B = static_cast<int>(q->shape[0]);
  s.Sq = static_cast<int>(q->shape[1]);
  s.H = static_cast<int>(q->shape[2]);
  s.D = static_cast<int>(q->shape[3]);
  s.Skv = static_cast<int>(k->shape[1]);
  if (q->shape[0] < 0 || q->shape[1] < 0 || q->shape[2] < 0 || k->shape[1] < 0 || q->shape[1] > (1ll << 30) ||
      k->shape[1] > (1ll << 30) || q->shape[0] > 65535 || q->shape[2] > 65535)
    return fail(ST_ERR_SHAPE, "sizes out of range");
  if (s.D != kD) return fail(ST_ERR_UNSUPPORTED, "head dimension %d is not supported (this build handles D=128)", s.D);
  st_status st;
  const unsigned qk_types = bit(ST_BF16) | bit(ST_F16) | bit(ST_F32);
  const unsigned v_types = bit(ST_BF16) | bit(ST_F16) | bit(ST_F32);
  if ((st = check_bshd(q, "q", s.B, s.Sq, s.H, s.D, qk_types, &P->q)) != ST_OK) return st;
  // grouped K/V heads: k and v carry H_kv heads, H a multiple of H_kv
  s.Hkv = static_cast<int>(k->shape[2]);
  if (s.H == 0 ? k->shape[2] != 0 : (k->shape[2] < 1 || k->shape[2] > 65535 || s.H % s.Hkv != 0))
    return fail(ST_ERR_SHAPE, "k has %lld heads: the K/V head count must divide H=%d", (long long)k->shape[2], s.H);
  if ((st = check_bshd(k, "k", s.B, s.Skv, s.Hkv, s.D, qk_types, &P->k)) != ST_OK) return st;
  if ((st = check_bshd(v, "v", s.B, s.Skv, s.Hkv, s.D, v_types, &P->v)) != ST_OK) return st;
  // the MMA operands take v's 16-bit type; 16-bit q/k must have it already
  // (they are staged as raw operand rows), fp32 q/k are cast to it on load;
  // fp32 v (with fp32 q/k) selects the exact-fp32 kernels
  if (q->dtype != k->dtype) return fail(ST_ERR_DTYPE, "q and k must have the same dtype");
  if (q->dtype != ST_F32 && q->dtype != v->dtype)
    return fail(ST_ERR_DTYPE, "16-bit q/k must have v's dtype (or be fp32, cast on load)");
  P->f32 = v->dtype == ST_F32;
  if (!rope) return fail(ST_ERR_INVALID_ARG, "rope is NULL");
  if (rope->cos || rope->sin) {  // the pages' table form
    if (rope->ids || rope->ids_k) return fail(ST_ERR_INVALID_ARG, "rope: give either ids or cos/sin tables, not both");
    if ((st = check_tables(rope->cos, rope->sin, "rope.cos/sin", s.B, s.Sq, &P->ids_q)) != ST_OK) return st;
    if (rope->cos_k || rope->sin_k) {
      if ((st = check_tables(rope->cos_k, rope->sin_k, "rope.cos_k/sin_k", s.B, s.Skv, &P->ids_k)) != ST_OK) return st;
      P->separate_k_table = true;
    } else {
      if (s.Sq != s.Skv) return fail(ST_ERR_INVALID_ARG, "rope.cos_k/sin_k are required when S_q != S_kv");
      P->ids_k = P->ids_q;
    }
  } else {
    if (rope->cos_k || rope->sin_k) return fail(ST_ERR_INVALID_ARG, "rope.cos_k/sin_k need rope.cos/sin");
    if (rope->n_axes < 1 || rope->n_axes > 8) return fail(ST_ERR_INVALID_ARG, "rope.n_axes must be 1..8");
    int dsum = 0;
    for (int a = 0; a < rope->n_axes; ++a) {
      if (rope->axes_dim[a] <= 0 || (rope->axes_dim[a] & 1))
        return fail(ST_ERR_INVALID_ARG, "rope.axes_dim[%d]=%d must be positive and even", a, rope->axes_dim[a]);
      dsum += rope->axes_dim[a];
    }
    if (dsum != s.D) return fail(ST_ERR_INVALID_ARG, "rope axes sum to %d, expected D=%d", dsum, s.D);
    if (!(rope->theta > 0.0) || !std::isfinite(rope->theta)) return fail(ST_ERR_INVALID_ARG, "rope.theta must be > 0");
    if ((st = check_ids(rope->ids, "rope.ids", s.B, s.Sq, rope->n_axes, &P->ids_q)) != ST_OK) return st;
    if (rope->ids_k) {
      if ((st = check_ids(rope->ids_k, "rope.ids_k", s.B, s.Skv, rope->n_axes, &P->ids_k)) != ST_OK) return st;
      P->separate_k_table = true;
    } else {
      if (s.Sq != s.Skv) return fail(ST_ERR_INVALID_ARG, "rope.ids_k is required when S_q != S_kv");
      P->ids_k = P->ids_q;
    }
  }
  if (mask && causal) return fail(ST_ERR_INVALID_ARG, "mask and causal cannot be combined");
  if (mask) {
    if (mask->ndim != 4) return fail(ST_ERR_SHAPE, "mask must be 4-D [B|1,H|1,S_q|1,S_kv]");
    const int64_t want[4] = {s.B, s.H, s.Sq, s.Skv};
    for (int a = 0; a < 3; ++a)
      if (!(mask->shape[a] == 1 || mask->shape[a] == want[a]))
        return fail(ST_ERR_SHAPE, "mask dim %d is %lld, expected 1 or %lld", a, (long long)mask->shape[a],
                    (long long)want[a]);
    if (mask->shape[3] != s.Skv) return fail(ST_ERR_SHAPE, "mask last dim must equal S_kv=%d", s.Skv);
    if (mask->dtype == ST_BOOL) P->mask_kind = kMaskBool;
    else if (mask->dtype == ST_F32) P->mask_kind = kMaskF32;
    else if (mask->dtype == ST_BF16) P->mask_kind = kMaskBF16;
    else return fail(ST_ERR_DTYPE, "mask must be bool, fp32 or bf16");
    if (s.Skv > 1 && mask->stride[3] != 1) return fail(ST_ERR_ALIGN, "mask must have unit stride on S_kv");
    if (!mask->data && (int64_t)s.B * s.H * s.Sq * s.Skv > 0) return fail(ST_ERR_INVALID_ARG, "mask data is NULL");
    P->Bm = static_cast<int>(mask->shape[0]);
    P->Hm = static_cast<int>(mask->shape[1]);
    P->Sqm = static_cast<int>(mask->shape[2]);
    P->m_sb = P->Bm > 1 ? mask->stride[0] : 0;
    P->m_sh = P->Hm > 1 ? mask->stride[1] : 0;
    P->m_sq = P->Sqm > 1 ? mask->stride[2] : 0;
  }
  P->sh = s;
  P->nQt = (s.Sq + kTile - 1) / kTile;
  P->nKt = (s.Skv + kTile - 1) / kTile;
  P->nQtm = P->Sqm > 1 ? P->nQt : 1;

  size_t off = 0;
  P->off_ctrl = off;
  off += 256;
  P->off_tab_q = off;
  off = align_up(off + (size_t)P->ids_q.Bt * s.Sq * kPairs * sizeof(float2), 256);
  P->off_tab16_q = off;
  off = align_up(off + (size_t)P->ids_q.Bt * s.Sq * kPairs * sizeof(__half2), 256);
  P->off_tab_k = P->off_tab_q;
  P->off_tab16_k = P->off_tab16_q;
  if (P->separate_k_table) {
    P->off_tab_k = off;
    off = align_up(off + (size_t)P->ids_k.Bt * s.Skv * kPairs * sizeof(float2), 256);
    P->off_tab16_k = off;
    off = align_up(off + (size_t)P->ids_k.Bt * s.Skv * kPairs * sizeof(__half2), 256);
  }
  if (P->mask_kind == kMaskBool) {
    P->off_flags = off;
    off = align_up(off + (size_t)P->Bm * P->Hm * P->nQtm * P->nKt, 256);
  }
  P->fwd_base = off;
  if (!P->f32 && P->nKt > 0) {
    // K' tiles shared between the forward's CTAs: publication flags
    // [B, H_kv, nKt] and the tiles [B, S_kv, H_kv, D] in the operand type
    P->kcache = true;
    P->off_kflags = off;
    off = align_up(off + (size_t)s.B * s.Hkv * P->nKt * sizeof(uint32_t), 256);
    P->off_kcache = off;
    off = align_up(off + (size_t)s.B * s.Skv * s.Hkv * kD * 2, 256);
  }
  if (for_backward) {
    P->off_delta = off;
    off = align_up(off + (size_t)s.B * s.H * s.Sq * sizeof(float), 256);
    P->off_dqacc = off;
    if (!P->f32) off = align_up(off + (size_t)s.B * s.Sq * s.H * kD * sizeof(float), 256);
    P->n_dwk = s.B * s.Hkv * P->nKt * 4;  // per backward CTA (key tile, K/V head, batch) and 32-row quarter
    if (P->f32) P->n_dwk = s.B * s.Hkv * ((s.Skv + kF32Tile - 1) / kF32Tile);  // per fp32 key tile
    P->off_dwk = off;
    off = align_up(off + (size_t)P->n_dwk * kD * sizeof(float), 256);
    P->n_dwq = static_cast<int>(((int64_t)s.B * s.Sq * s.H + kPostBlockRows - 1) / kPostBlockRows);
    if (P->f32) P->n_dwq = s.B * s.H * ((s.Sq + kF32Tile - 1) / kF32Tile);  // per fp32 query tile
    P->off_dwq = off;
    off = align_up(off + (size_t)P->n_dwq * kD * sizeof(float), 256);
    P->off_dwscratch = off;
    off = align_up(off + (size_t)2 * dw_reduce_blocks(P->n_dwq, P->n_dwk) * kD * sizeof(float), 256);
    if (!P->f32) {  // Q' rows [B, S_q, H, D] in the 16-bit operand type, left by the forward
      P->off_qp = off;
      off = align_up(off + (size_t)s.B * s.Sq * s.H * kD * 2, 256);
    }
  }
  P->total = off;
  return ST_OK;
}

void fill_common(const Plan& P, const st_tensor* qw, const st_tensor* kw, float eps, int causal, float scale,
                 uint8_t* ws, const Dev& dev, Common* c) {
  memset(c, 0, sizeof(*c));
  c->q = P.q;
  c->k = P.k;
  c->v = P.v;
  c->wq = static_cast<const float*>(qw->data);
  c->wk = static_cast<const float*>(kw->data);
  c->eps = eps;
  c->tab_q = reinterpret_cast<const float2*>(ws + P.off_tab_q);
  c->tab_k = reinterpret_cast<const float2*>(ws + P.off_tab_k);
  c->tab16_q = reinterpret_cast<const __half2*>(ws + P.off_tab16_q);
  c->tab16_k = reinterpret_cast<const __half2*>(ws + P.off_tab16_k);
  c->tab_q_sb = P.ids_q.Bt > 1 ? (int64_t)P.sh.Sq * kPairs : 0;
  c->tab_k_sb = P.ids_k.Bt > 1 ? (int64_t)P.sh.Skv * kPairs : 0;
  c->mask_kind = P.mask_kind;
  c->m_sb = P.m_sb;
  c->m_sh = P.m_sh;
  c->m_sq = P.m_sq;
  if (P.mask_kind == kMaskBool) {
    c->flags = ws + P.off_flags;
    c->mask_any_false = reinterpret_cast<const unsigned*>(ws + P.off_ctrl) + kCtrlAnyFalse;
    c->f_sb = P.Bm > 1 ? (int64_t)P.Hm * P.nQtm * P.nKt : 0;
    c->f_sh = P.Hm > 1 ? (int64_t)P.nQtm * P.nKt : 0;
    c->f_sq = P.nQtm > 1 ? P.nKt : 0;
  }
  c->causal = causal ? 1 : 0;
  c->f16 = P.v.dt == kDtF16 ? 1 : 0;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(kD));
  c->scale = sc;
  c->scale_log2 = sc * kLog2e;
  c->B = P.sh.B;
  c->H = P.sh.H;
  c->Hkv = P.sh.Hkv;
  c->group = P.sh.Hkv > 0 ? P.sh.H / P.sh.Hkv : 1;
  c->Sq = P.sh.Sq;
  c->Skv = P.sh.Skv;
  c->nQt = P.nQt;
  c->nKt = P.nKt;
  c->status = dev.status;
  c->counters = dev.counters;
  c->wait_budget = wait_budget();
}

void fill_table(const Ids& ids, const st_rope* rope, float2* out, __half2* out16, unsigned* ctrl, TableParams* t) {
  memset(t, 0, sizeof(*t));
  t->Bt = ids.Bt;
  t->S = ids.S;
  t->out = out;
  t->out16 = out16;
  t->ctrl = ctrl;
  if (ids.table) {
    const st_tensor *c = ids.t, *sn = ids.sin;
    const int o = c->ndim - 2;
    t->cos = c->data;
    t->sin = sn->data;
    t->tab_dtype = c->dtype;
    t->c_sb = (c->ndim == 3 && ids.Bt > 1) ? c->stride[0] : 0;
    t->c_ss = c->stride[o];
    t->c_sd = c->stride[o + 1];
    t->s_sb = (sn->ndim == 3 && ids.Bt > 1) ? sn->stride[0] : 0;
    t->s_ss = sn->stride[o];
    t->s_sd = sn->stride[o + 1];
    return;
  }
  t->ids = ids.t->data;
  t->ids_f32 = ids.t->dtype == ST_F32;
  t->i_sb = ids.t->stride[0];
  t->i_ss = ids.t->stride[1];
  t->i_sa = ids.t->stride[2];
  int pair = 0;
  for (int a = 0; a < rope->n_axes; ++a) {
    const int da = rope->axes_dim[a];
    for (int j = 0; j < da / 2; ++j, ++pair) {
      t->omega[pair] = std::pow(rope->theta, -2.0 * j / static_cast<double>(da));
      t->axis_of[pair] = a;
    }
  }
}

st_status cuda_check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(ST_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ST_OK;
}

// Rotary tables and mask tile classes: the first launches of a call.
st_status launch_prelude(const Plan& P, const st_rope* rope, const st_tensor* mask, uint8_t* ws, const Dev& dev,
                         cudaStream_t stream, bool zero_kflags = false) {
  unsigned* ctrl = reinterpret_cast<unsigned*>(ws + P.off_ctrl);
  TableParams t;
  fill_table(P.ids_q, rope, reinterpret_cast<float2*>(ws + P.off_tab_q), reinterpret_cast<__half2*>(ws + P.off_tab16_q),
             ctrl, &t);
  if (zero_kflags) {  // the forward's K' publication flags start lowered
    t.zero = reinterpret_cast<unsigned*>(ws + P.off_kflags);
    t.n_zero = (int64_t)P.sh.B * P.sh.Hkv * P.nKt;
  }
  st_status st = cuda_check(launch_counted(ST_K_TABLE, stream, [&] { return launch_table(t, stream); }), "table kernel launch");
  if (st != ST_OK) return st;
  if (P.separate_k_table) {
    fill_table(P.ids_k, rope, reinterpret_cast<float2*>(ws + P.off_tab_k),
               reinterpret_cast<__half2*>(ws + P.off_tab16_k), nullptr, &t);
    if ((st = cuda_check(launch_counted(ST_K_TABLE, stream, [&] { return launch_table(t, stream); }), "table kernel launch")) != ST_OK) return st;
  }
  if (P.mask_kind == kMaskBool && P.nKt > 0 && P.nQt > 0) {
    ClassifyParams cp;
    memset(&cp, 0, sizeof(cp));
    cp.mask = static_cast<const uint8_t*>(mask->data);
    cp.m_sb = P.m_sb;
    cp.m_sh = P.m_sh;
    cp.m_sq = P.m_sq;
    cp.Bm = P.Bm;
    cp.Hm = P.Hm;
    cp.Sqm = P.Sqm > 1 ? P.sh.Sq : 1;
    cp.Skv = P.sh.Skv;
    cp.nQtm = P.nQtm;
    cp.nKt = P.nKt;
    cp.flags = ws + P.off_flags;
    cp.ctrl = ctrl;
    cp.counters = dev.counters;
    if ((st = cuda_check(launch_counted(ST_K_CLASSIFY, stream, [&] { return launch_classify(cp, stream); }), "mask classify launch")) != ST_OK) return st;
  }
  return ST_OK;
}

st_status check_workspace(const Plan& P, void* ws, size_t bytes) {
  if (bytes < P.total) return fail(ST_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu required", bytes, P.total);
  if (P.total > 0 && !ws) return fail(ST_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(ST_ERR_ALIGN, "workspace must be 256-byte aligned");
  return ST_OK;
}

st_status check_out(const st_tensor* t, const char* name, int B, int S, int H, int dtype, RowTensor* rt) {
  return check_bshd(t, name, B, S, H, kD, bit(dtype), rt);
}

// The encoder is a driver call and needs a context current on the calling
// thread. A thread that has made no runtime call yet (an autograd worker
// thread running the backward) has none: cudaSetDevice binds the current
// device's primary context to it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaSetDevice(dev);
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 4-D tiled map over a bf16, fp16 or fp32 [B, S, H, D] tensor for boxes of
// 128 bytes (64 16-bit or 32 fp32 columns) x box_rows rows with 128-byte
// swizzle. The two
// middle dims are ordered by stride (s before h when the sequence stride is the
// smaller one, as in a BHSD view).
st_status encode_rows_map(const st_tensor* t, CUtensorMap* map, int* s_first, int box_rows = kTile) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ST_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int64_t B = t->shape[0], S = t->shape[1], H = t->shape[2];
  const bool f32 = t->dtype == ST_F32;
  const int64_t eb = f32 ? 4 : 2;
  // strides in bytes; a size-1 dim gets the packed stride (any valid value works)
  int64_t ss = S > 1 ? t->stride[1] * eb : H * kD * eb;
  int64_t sh = H > 1 ? t->stride[2] * eb : kD * eb;
  int64_t sb = B > 1 ? t->stride[0] * eb : S * H * kD * eb;
  if (ss == 0) ss = H * kD * eb;
  if (sh == 0) sh = kD * eb;
  if (sb == 0) sb = S * H * kD * eb;
  *s_first = ss < sh;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4] = {f32 ? 32u : 64u, 1, 1, 1}, es[4] = {1, 1, 1, 1};
  dims[0] = kD;
  if (*s_first) {
    dims[1] = S; dims[2] = H; strides[0] = ss; strides[1] = sh; box[1] = box_rows;
  } else {
    dims[1] = H; dims[2] = S; strides[0] = sh; strides[1] = ss; box[2] = box_rows;
  }
  dims[3] = B;
  strides[2] = sb;
  const CUtensorMapDataType ty = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : (t->dtype == ST_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  CUresult r = enc(map, ty, 4, t->data, dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ST_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the layout (error %d)", (int)r);
  return ST_OK;
}

// 2-D tiled map over an fp32 rotary table [rows, 64] float2 (cos, sin) seen as
// [rows, 128] floats, for 32-float x 128-row boxes with 128-byte swizzle: the
// backward's epilogue stages a key tile's table rows with it.
st_status encode_table_map(const float2* tab, int64_t rows, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ST_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
  cuuint32_t box[2] = {32, kTile}, es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float2*>(tab), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ST_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the rotary table (error %d)", (int)r);
  return ST_OK;
}

// 4-D tiled map over the fp32 dQ accumulator [B, S_q, H, D] (contiguous) as
// (d, h, s, b) for 32-column x 64-row boxes with 128-byte swizzle: the target
// of the backward kernel's bulk reductions (one box per 32 head dims of a
// 64-query half of a query tile).
st_status encode_dq_acc_map(float* dq_acc, int B, int Sq, int H, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ST_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t row = (cuuint64_t)kD * 4;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)Sq, (cuuint64_t)B};
  cuuint64_t strides[3] = {row, row * H, row * H * Sq};
  cuuint32_t box[4] = {32, 1, kTile / 2, 1}, es[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq_acc, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ST_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the dq accumulator (error %d)", (int)r);
  return ST_OK;
}

// 4-D tiled map over contiguous operand rows [B, S, H, D] of the workspace (the
// 16-bit operand type) as (d, h, s, b), for 64-column x box_rows boxes with
// 128-byte swizzle: the Q' rows (the forward stores its tiles, each backward
// CTA of a pair loads half of a tile) and the forward's shared K' tiles.
st_status encode_operand_rows_map(uint8_t* base, int B, int S, int H, bool f16, int box_rows, CUtensorMap* map) {
  st_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = base;
  t.dtype = f16 ? ST_F16 : ST_BF16;
  t.ndim = 4;
  t.shape[0] = B; t.shape[1] = S; t.shape[2] = H; t.shape[3] = kD;
  t.stride[3] = 1; t.stride[2] = kD; t.stride[1] = (int64_t)H * kD; t.stride[0] = (int64_t)S * H * kD;
  int s_first = 0;
  st_status st = encode_rows_map(&t, map, &s_first, box_rows);
  if (st == ST_OK && s_first) return fail(ST_ERR_UNSUPPORTED, "unexpected operand-row map order");
  return st;
}

// The forward's launches (tables, mask tile classes, attention) on a
// validated call, with `ws` the workspace (or the built-in scratch). With
// `qp` non-null the attention kernel also stores its Q' tiles there.
st_status enqueue_forward(const Plan& P, const st_tensor* q, const st_tensor* k, const st_tensor* v,
                          const st_tensor* q_norm_w, const st_tensor* k_norm_w, float eps, const st_rope* rope,
                          const st_tensor* mask, int causal, float scale, st_tensor* o, const RowTensor& ro,
                          st_tensor* lse, uint8_t* ws, uint8_t* qp, float* dq_zero, bool kcache,
                          cudaStream_t stream) {
  st_status st;
  Dev dev;
  if ((st = device_globals(&dev)) != ST_OK) return st;
  if (P.f32) {
    F32Params fp;
    memset(&fp, 0, sizeof(fp));
    fill_common(P, q_norm_w, k_norm_w, eps, causal, scale, ws, dev, &fp.c);
    fp.c.mask = mask ? mask->data : nullptr;
    fp.o = static_cast<float*>(o->data);
    fp.o_sb = ro.sb; fp.o_ss = ro.ss; fp.o_sh = ro.sh;
    fp.lse = static_cast<float*>(lse->data);
    if ((st = launch_prelude(P, rope, mask, ws, dev, stream)) != ST_OK) return st;
    return cuda_check(launch_counted(ST_K_FWD, stream, [&] { return launch_f32_fwd(fp, stream); }),
                      "fp32 forward kernel launch");
  }
  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  fill_common(P, q_norm_w, k_norm_w, eps, causal, scale, ws, dev, &fp.c);
  fp.c.mask = mask ? mask->data : nullptr;
  fp.o = o->data;
  fp.o_sb = ro.sb;
  fp.o_ss = ro.ss;
  fp.o_sh = ro.sh;
  fp.o_dt = ro.dt;
  fp.lse = static_cast<float*>(lse->data);
  if (P.nKt > 0 && (st = encode_rows_map(v, &fp.tmap_v, &fp.v_s_first)) != ST_OK) return st;
  fp.qk_tma = q->dtype != ST_F32 ? 1 : 0;
  if (fp.qk_tma) {
    if ((st = encode_rows_map(q, &fp.tmap_q, &fp.q_s_first)) != ST_OK) return st;
    if (P.nKt > 0 && (st = encode_rows_map(k, &fp.tmap_k, &fp.k_s_first)) != ST_OK) return st;
  }
  if (qp) {
    if ((st = encode_operand_rows_map(qp, P.sh.B, P.sh.Sq, P.sh.H, v->dtype == ST_F16, kTile, &fp.tmap_qp)) != ST_OK) return st;
    fp.save_qp = 1;
    fp.dq_zero = dq_zero;
  }
  kcache = kcache && P.kcache;
  if (kcache) {
    if ((st = encode_operand_rows_map(ws + P.off_kcache, P.sh.B, P.sh.Skv, P.sh.Hkv, v->dtype == ST_F16, kTile,
                                      &fp.tmap_kc)) != ST_OK)
      return st;
    fp.kflags = reinterpret_cast<uint32_t*>(ws + P.off_kflags);
    fp.kcache = 1;
  }
  if ((st = launch_prelude(P, rope, mask, ws, dev, stream, kcache)) != ST_OK) return st;
  return cuda_check(launch_counted(ST_K_FWD, stream, [&] { return launch_fwd(fp, stream); }), "forward kernel launch");
}

}  // namespace

extern "C" {

size_t st_rope_attn_workspace_size(const st_tensor* q, const st_tensor* k, const st_tensor* v,
                                   const st_tensor* mask, int causal, const st_rope* rope, int for_backward) {
  Plan P;
  if (plan_call(q, k, v, mask, causal, rope, for_backward, &P) != ST_OK) return 0;
  return P.total;
}

st_status st_rope_attn_fwd(const st_tensor* q, const st_tensor* k, const st_tensor* v, const st_tensor* q_norm_w,
                           const st_tensor* k_norm_w, float eps, const st_rope* rope, const st_tensor* mask,
                           int causal, float scale, st_tensor* o, st_tensor* lse, void* workspace,
                           size_t workspace_bytes, void* stream_) {
  t_err.clear();
  Plan P;
  st_status st = plan_call(q, k, v, mask, causal, rope, 0, &P);
  if (st != ST_OK) return st;
  const Shape& s = P.sh;
  if ((st = check_vec(q_norm_w, "q_norm_w", kD)) != ST_OK) return st;
  if ((st = check_vec(k_norm_w, "k_norm_w", kD)) != ST_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ST_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!std::isfinite(scale)) return fail(ST_ERR_INVALID_ARG, "scale must be finite");
  RowTensor ro;
  if ((st = check_out(o, "o", s.B, s.Sq, s.H, v->dtype, &ro)) != ST_OK) return st;
  if (!lse || lse->ndim != 3 || lse->shape[0] != s.B || lse->shape[1] != s.H || lse->shape[2] != s.Sq)
    return fail(ST_ERR_SHAPE, "lse must be [B,H,S_q] = [%d,%d,%d]", s.B, s.H, s.Sq);
  if (lse->dtype != ST_F32) return fail(ST_ERR_DTYPE, "lse must be fp32");
  if ((int64_t)s.B * s.H * s.Sq > 0 &&
      (!lse->data || lse->stride[2] != 1 || lse->stride[1] != s.Sq || lse->stride[0] != (int64_t)s.H * s.Sq))
    return fail(ST_ERR_ALIGN, "lse must be contiguous");
  if ((st = check_workspace(P, workspace, workspace_bytes)) != ST_OK) return st;
  if ((int64_t)s.B * s.H * s.Sq == 0) {
    ++h_fwd_calls;
    return ST_OK;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // a workspace that can also serve the backward receives the Q' rows, which
  // a backward reusing it reads instead of normalising and rotating q again
  // and a zeroed dQ' accumulator
  uint8_t* qp = nullptr;
  float* dq_zero = nullptr;
  if (!P.f32) {
    Plan PB;
    if (plan_call(q, k, v, mask, causal, rope, 1, &PB) == ST_OK && workspace_bytes >= PB.total) {
      qp = static_cast<uint8_t*>(workspace) + PB.off_qp;
      dq_zero = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + PB.off_dqacc);
    }
  }
  if ((st = enqueue_forward(P, q, k, v, q_norm_w, k_norm_w, eps, rope, mask, causal, scale, o, ro, lse,
                            static_cast<uint8_t*>(workspace), qp, dq_zero, true, stream)) != ST_OK)
    return st;
  ++h_fwd_calls;
  if (q->dtype == ST_F32 && !P.f32) ++h_mixed;
  return ST_OK;
}

st_status st_rope_attn_bwd(const st_tensor* q, const st_tensor* k, const st_tensor* v, const st_tensor* q_norm_w,
                           const st_tensor* k_norm_w, float eps, const st_rope* rope, const st_tensor* mask,
                           int causal, float scale, const st_tensor* o, const st_tensor* lse, const st_tensor* d_o,
                           st_tensor* dq, st_tensor* dk, st_tensor* dv, st_tensor* d_q_norm_w,
                           st_tensor* d_k_norm_w, void* workspace, size_t workspace_bytes, void* stream_) {
  t_err.clear();
  Plan P;
  st_status st = plan_call(q, k, v, mask, causal, rope, 1, &P);
  if (st != ST_OK) return st;
  const Shape& s = P.sh;
  if ((st = check_vec(q_norm_w, "q_norm_w", kD)) != ST_OK) return st;
  if ((st = check_vec(k_norm_w, "k_norm_w", kD)) != ST_OK) return st;
  if ((st = check_vec(d_q_norm_w, "d_q_norm_w", kD)) != ST_OK) return st;
  if ((st = check_vec(d_k_norm_w, "d_k_norm_w", kD)) != ST_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ST_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!std::isfinite(scale)) return fail(ST_ERR_INVALID_ARG, "scale must be finite");
  RowTensor ro, rdo, rdq, rdk, rdv;
  if ((st = check_out(o, "o", s.B, s.Sq, s.H, v->dtype, &ro)) != ST_OK) return st;
  if ((st = check_out(d_o, "d_o", s.B, s.Sq, s.H, v->dtype, &rdo)) != ST_OK) return st;
  if ((st = check_out(dq, "dq", s.B, s.Sq, s.H, q->dtype, &rdq)) != ST_OK) return st;
  if ((st = check_out(dk, "dk", s.B, s.Skv, s.Hkv, k->dtype, &rdk)) != ST_OK) return st;
  if ((st = check_out(dv, "dv", s.B, s.Skv, s.Hkv, v->dtype, &rdv)) != ST_OK) return st;
  if (!lse || lse->ndim != 3 || lse->shape[0] != s.B || lse->shape[1] != s.H || lse->shape[2] != s.Sq)
    return fail(ST_ERR_SHAPE, "lse must be [B,H,S_q] = [%d,%d,%d]", s.B, s.H, s.Sq);
  if (lse->dtype != ST_F32) return fail(ST_ERR_DTYPE, "lse must be fp32");
  if ((int64_t)s.B * s.H * s.Sq > 0 &&
      (!lse->data || lse->stride[2] != 1 || lse->stride[1] != s.Sq || lse->stride[0] != (int64_t)s.H * s.Sq))
    return fail(ST_ERR_ALIGN, "lse must be contiguous");
  if ((st = check_workspace(P, workspace, workspace_bytes)) != ST_OK) return st;
  if ((int64_t)s.B * s.H == 0) {
    ++h_bwd_calls;
    return ST_OK;
  }
  Dev dev;
  if ((st = device_globals(&dev)) != ST_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdParams bp;
  memset(&bp, 0, sizeof(bp));
  if (P.nKt > 0 && !P.f32) {
    if ((st = encode_rows_map(v, &bp.tmap_v, &bp.v_s_first)) != ST_OK) return st;
    if ((int64_t)s.B * s.Sq * s.H > 0 && (st = encode_rows_map(d_o, &bp.tmap_do, &bp.do_s_first, kTile)) != ST_OK)
      return st;
    bp.qk_tma = q->dtype != ST_F32 ? 1 : 0;
    // raw k rows: the prologue's TMA source (bf16) and the epilogue's (both dtypes)
    if ((st = encode_rows_map(k, &bp.tmap_k, &bp.k_s_first)) != ST_OK) return st;
    // the Q' rows of the workspace, 64-row boxes (each CTA of a pair loads half a tile)
    if ((int64_t)s.B * s.Sq * s.H > 0 &&
        (st = encode_operand_rows_map(ws + P.off_qp, s.B, s.Sq, s.H, v->dtype == ST_F16, kTile / 2, &bp.tmap_q)) != ST_OK)
      return st;
    if ((st = encode_table_map(reinterpret_cast<const float2*>(ws + P.off_tab_k), (int64_t)P.ids_k.Bt * s.Skv,
                               &bp.tmap_tab_k)) != ST_OK)
      return st;
  }
  // the forward's tables and mask tile classes, when the caller says the
  // workspace holds them (the pre kernel then clears the control words that
  // the table kernel would have cleared)
  const bool reuse = rope->reuse_tables != 0 && (int64_t)s.B * s.Sq * s.H > 0;
  if (!reuse && (st = launch_prelude(P, rope, mask, ws, dev, stream)) != ST_OK) return st;
  if (reuse && P.kcache && P.nKt > 0) {
    // the forward on this workspace published every K' tile that a query tile needs
    if ((st = encode_operand_rows_map(ws + P.off_kcache, s.B, s.Skv, s.Hkv, v->dtype == ST_F16, kTile,
                                      &bp.tmap_kc)) != ST_OK)
      return st;
    bp.kp_ready = 1;
    bp.kflags = reinterpret_cast<const uint32_t*>(ws + P.off_kflags);
  }
  if (!reuse && !P.f32 && P.nKt > 0 && (int64_t)s.B * s.Sq * s.H > 0) {
    // no forward left its Q' rows in this workspace: build them
    QPrimeParams qpp;
    memset(&qpp, 0, sizeof(qpp));
    qpp.q = P.q;
    qpp.tab = reinterpret_cast<const float2*>(ws + P.off_tab_q);
    qpp.tab16 = reinterpret_cast<const __half2*>(ws + P.off_tab16_q);
    qpp.tab_sb = P.ids_q.Bt > 1 ? (int64_t)s.Sq * kPairs : 0;
    qpp.w = static_cast<const float*>(q_norm_w->data);
    qpp.eps = eps;
    qpp.out = ws + P.off_qp;
    qpp.f16 = v->dtype == ST_F16 ? 1 : 0;
    qpp.B = s.B; qpp.H = s.H; qpp.Sq = s.Sq;
    if ((st = cuda_check(launch_counted(ST_K_QPRIME, stream, [&] { return launch_qprime(qpp, stream); }),
                         "Q' row kernel launch")) != ST_OK)
      return st;
  }

  float* delta = reinterpret_cast<float*>(ws + P.off_delta);
  float* dq_acc = P.f32 ? nullptr : reinterpret_cast<float*>(ws + P.off_dqacc);  // the fp32 path needs none
  if ((int64_t)s.B * s.Sq * s.H > 0) {
    PreParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.o = o->data;
    pp.o_sb = ro.sb; pp.o_ss = ro.ss; pp.o_sh = ro.sh; pp.o_dt = ro.dt;
    pp.dout = d_o->data;
    pp.do_sb = rdo.sb; pp.do_ss = rdo.ss; pp.do_sh = rdo.sh;
    pp.delta = delta;
    pp.dq_acc = reuse ? nullptr : dq_acc;  // a reused workspace: the forward zeroed it
    pp.ctrl = reinterpret_cast<unsigned*>(ws + P.off_ctrl);
    pp.B = s.B; pp.H = s.H; pp.Sq = s.Sq;
    if ((st = cuda_check(launch_counted(ST_K_BWD_PRE, stream, [&] { return launch_bwd_pre(pp, stream); }), "backward pre launch")) != ST_OK) return st;
  }
  if (P.f32) {
    // exact fp32: a kernel over key tiles (dk, dv), one over query tiles (dq)
    F32Params fp;
    memset(&fp, 0, sizeof(fp));
    fill_common(P, q_norm_w, k_norm_w, eps, causal, scale, ws, dev, &fp.c);
    fp.c.mask = mask ? mask->data : nullptr;
    fp.lse_in = static_cast<const float*>(lse->data);
    fp.delta = delta;
    fp.dout = static_cast<const float*>(d_o->data);
    fp.do_sb = rdo.sb; fp.do_ss = rdo.ss; fp.do_sh = rdo.sh;
    fp.dq = static_cast<float*>(dq->data); fp.dq_sb = rdq.sb; fp.dq_ss = rdq.ss; fp.dq_sh = rdq.sh;
    fp.dk = static_cast<float*>(dk->data); fp.dk_sb = rdk.sb; fp.dk_ss = rdk.ss; fp.dk_sh = rdk.sh;
    fp.dv = static_cast<float*>(dv->data); fp.dv_sb = rdv.sb; fp.dv_ss = rdv.ss; fp.dv_sh = rdv.sh;
    fp.dwq_part = reinterpret_cast<float*>(ws + P.off_dwq);
    fp.dwk_part = reinterpret_cast<float*>(ws + P.off_dwk);
    if (s.Skv > 0 && (st = cuda_check(launch_counted(ST_K_BWD, stream, [&] { return launch_f32_bwd_kv(fp, stream); }),
                                      "fp32 backward (keys) launch")) != ST_OK)
      return st;
    if ((int64_t)s.B * s.Sq * s.H > 0 &&
        (st = cuda_check(launch_counted(ST_K_DQ_POST, stream, [&] { return launch_f32_bwd_q(fp, stream); }),
                         "fp32 backward (queries) launch")) != ST_OK)
      return st;
  }
  if (P.nKt > 0 && !P.f32) {
    fill_common(P, q_norm_w, k_norm_w, eps, causal, scale, ws, dev, &bp.c);
    bp.c.mask = mask ? mask->data : nullptr;
    bp.dout = d_o->data;
    bp.do_sb = rdo.sb; bp.do_ss = rdo.ss; bp.do_sh = rdo.sh;
    bp.lse = static_cast<const float*>(lse->data);
    bp.delta = delta;
    bp.dq_acc = dq_acc;
    if ((int64_t)s.B * s.Sq * s.H > 0 && (st = encode_dq_acc_map(dq_acc, s.B, s.Sq, s.H, &bp.tmap_dq)) != ST_OK)
      return st;
    bp.dv = dv->data; bp.dv_sb = rdv.sb; bp.dv_ss = rdv.ss; bp.dv_sh = rdv.sh; bp.dv_dt = rdv.dt;
    bp.dk = dk->data; bp.dk_sb = rdk.sb; bp.dk_ss = rdk.ss; bp.dk_sh = rdk.sh; bp.dk_dt = rdk.dt;
    // the epilogue stores dv (and 16-bit dk) rows by TMA
    if ((st = encode_rows_map(dv, &bp.tmap_dv, &bp.dv_s_first)) != ST_OK) return st;
    if (bp.qk_tma && (st = encode_rows_map(dk, &bp.tmap_dk, &bp.dk_s_first)) != ST_OK) return st;
    bp.dwk_part = reinterpret_cast<float*>(ws + P.off_dwk);
    if ((st = cuda_check(launch_counted(ST_K_BWD, stream, [&] { return launch_bwd(bp, stream); }), "backward kernel launch")) != ST_OK) return st;
  }
  if ((int64_t)s.B * s.Sq * s.H > 0 && !P.f32) {
    PostParams pq;
    memset(&pq, 0, sizeof(pq));
    pq.dq_acc = dq_acc;
    pq.q = P.q;
    pq.tab_q = reinterpret_cast<const float2*>(ws + P.off_tab_q);
    pq.tab_q_sb = P.ids_q.Bt > 1 ? (int64_t)s.Sq * kPairs : 0;
    pq.wq = static_cast<const float*>(q_norm_w->data);
    pq.eps = eps;
    pq.dq = dq->data; pq.dq_sb = rdq.sb; pq.dq_ss = rdq.ss; pq.dq_sh = rdq.sh; pq.dq_dt = rdq.dt;
    pq.dwq_part = reinterpret_cast<float*>(ws + P.off_dwq);
    pq.B = s.B; pq.H = s.H; pq.Sq = s.Sq;
    if ((st = cuda_check(launch_counted(ST_K_DQ_POST, stream, [&] { return launch_dq_post(pq, stream); }), "dq post launch")) != ST_OK) return st;
  }
  DwParams dp;
  memset(&dp, 0, sizeof(dp));
  dp.dwq_part = reinterpret_cast<const float*>(ws + P.off_dwq);
  dp.dwk_part = reinterpret_cast<const float*>(ws + P.off_dwk);
  dp.n_q = (int64_t)s.B * s.Sq * s.H > 0 ? P.n_dwq : 0;
  dp.n_k = P.nKt > 0 ? P.n_dwk : 0;
  dp.scratch = reinterpret_cast<float*>(ws + P.off_dwscratch);
  dp.ctrl = reinterpret_cast<unsigned*>(ws + P.off_ctrl);
  dp.dwq = static_cast<float*>(d_q_norm_w->data);
  dp.dwk = static_cast<float*>(d_k_norm_w->data);
  if ((st = cuda_check(launch_counted(ST_K_DW, stream, [&] { return launch_dw_reduce(dp, stream); }), "weight-gradient reduce launch")) != ST_OK) return st;
  ++h_bwd_calls;
  if (q->dtype == ST_F32 && !P.f32) ++h_mixed;
  return ST_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward with built-in scratch, for callers that cannot allocate device
// memory (see st_rope_attn_fwd_noalloc in the header). The scratch is this
// file-scope array; host code never uses its name as an address: the device
// address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ST_NOALLOC_SCRATCH_BYTES];

namespace {

st_status noalloc_scratch_address(void** out) {
  static void* addr[64];
  static std::atomic<bool> ready[64];
  static std::mutex mu;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(ST_ERR_CUDA, "cudaGetDevice failed");
  if (!ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev].load(std::memory_order_relaxed)) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return fail(ST_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
      addr[dev] = p;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  *out = addr[dev];
  return ST_OK;
}

}  // namespace

extern "C" {

st_status st_rope_attn_fwd_noalloc(const st_tensor* q, const st_tensor* k, const st_tensor* v,
                                   const st_tensor* q_norm_w, const st_tensor* k_norm_w, float eps,
                                   const st_rope* rope, const st_tensor* mask, int causal, float scale,
                                   st_tensor* o, st_tensor* lse, void* stream_) {
  t_err.clear();
  Plan P;
  st_status st = plan_call(q, k, v, mask, causal, rope, 0, &P);
  if (st != ST_OK) return st;
  // the K' tile cache is used only when it fits as well
  if (P.fwd_base > ST_NOALLOC_SCRATCH_BYTES)
    return fail(ST_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch; the built-in scratch holds %u bytes "
                "(use st_rope_attn_fwd with a caller workspace)",
                P.fwd_base, (unsigned)ST_NOALLOC_SCRATCH_BYTES);
  const Shape& s = P.sh;
  if ((st = check_vec(q_norm_w, "q_norm_w", kD)) != ST_OK) return st;
  if ((st = check_vec(k_norm_w, "k_norm_w", kD)) != ST_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ST_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!std::isfinite(scale)) return fail(ST_ERR_INVALID_ARG, "scale must be finite");
  RowTensor ro;
  if ((st = check_out(o, "o", s.B, s.Sq, s.H, v->dtype, &ro)) != ST_OK) return st;
  if (!lse || lse->ndim != 3 || lse->shape[0] != s.B || lse->shape[1] != s.H || lse->shape[2] != s.Sq)
    return fail(ST_ERR_SHAPE, "lse must be [B,H,S_q] = [%d,%d,%d]", s.B, s.H, s.Sq);
  if (lse->dtype != ST_F32) return fail(ST_ERR_DTYPE, "lse must be fp32");
  if ((int64_t)s.B * s.H * s.Sq > 0 &&
      (!lse->data || lse->stride[2] != 1 || lse->stride[1] != s.Sq || lse->stride[0] != (int64_t)s.H * s.Sq))
    return fail(ST_ERR_ALIGN, "lse must be contiguous");
  if ((int64_t)s.B * s.H * s.Sq == 0) {
    ++h_fwd_calls;
    return ST_OK;
  }
  void* scratch = nullptr;
  if ((st = noalloc_scratch_address(&scratch)) != ST_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if ((st = enqueue_forward(P, q, k, v, q_norm_w, k_norm_w, eps, rope, mask, causal, scale, o, ro, lse,
                            static_cast<uint8_t*>(scratch), nullptr, nullptr, P.total <= ST_NOALLOC_SCRATCH_BYTES,
                            stream)) != ST_OK)
    return st;
  ++h_fwd_calls;
  if (q->dtype == ST_F32 && !P.f32) ++h_mixed;
  return ST_OK;
}

const char* st_last_error(void) { return t_err.c_str(); }

st_status st_get_stats(st_stats* out) {
  if (!out) return fail(ST_ERR_INVALID_ARG, "out is NULL");
  memset(out, 0, sizeof(*out));
  out->fwd_calls = h_fwd_calls.load();
  out->bwd_calls = h_bwd_calls.load();
  out->mixed_dtype_calls = h_mixed.load();
  Dev dev;
  st_status st = device_globals(&dev);
  if (st != ST_OK) return st;
  unsigned long long c[kNumCounters];
  if ((st = cuda_check(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) != ST_OK) return st;
  if ((st = cuda_check(cudaMemcpy(c, dev.counters, sizeof(c), cudaMemcpyDeviceToHost), "read counters")) != ST_OK)
    return st;
  out->mask_all_true_skipped = c[kCtrMaskAllTrue];
  out->tiles_skipped = c[kCtrTilesSkipped];
  out->tiles_total = c[kCtrTilesTotal];
  out->timeouts = c[kCtrTimeouts];
  out->kernel_launches = h_launches.load();
  return ST_OK;
}

st_status st_selftest_wait_timeout(long long budget_cycles, void* stream_) {
  if (budget_cycles < 1 || budget_cycles > (1ll << 34)) return fail(ST_ERR_INVALID_ARG, "budget out of range");
  Dev dev;
  st_status st = device_globals(&dev);
  if (st != ST_OK) return st;
  return cuda_check(launch_counted(ST_K_PROBE, static_cast<cudaStream_t>(stream_),
                                   [&] {
                                     return launch_wait_probe(dev.status, dev.counters, budget_cycles,
                                                              static_cast<cudaStream_t>(stream_));
                                   }),
                    "wait probe launch");
}

st_status st_timing_enable(int on) {
  g_timing.store(on != 0);
  return ST_OK;
}

st_status st_timing_read(st_kernel_times* out) {
  if (!out) return fail(ST_ERR_INVALID_ARG, "out is NULL");
  memset(out, 0, sizeof(*out));
  std::vector<TimedLaunch> done;
  {
    std::lock_guard<std::mutex> lk(g_tmu);
    done.swap(g_pending);
  }
  st_status st = ST_OK;
  for (const TimedLaunch& t : done) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(t.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.a, t.b);
    if (e != cudaSuccess && st == ST_OK) st = fail(ST_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
    if (t.kind >= 0 && t.kind < ST_K_COUNT) {
      out->launches[t.kind] += 1;
      out->ms[t.kind] += ms;
    }
  }
  std::lock_guard<std::mutex> lk(g_tmu);
  for (const TimedLaunch& t : done) {
    g_event_pool.push_back(t.a);
    g_event_pool.push_back(t.b);
  }
  return st;
}

void st_reset_stats(void) {
  h_launches = 0;
  h_fwd_calls = 0;
  h_bwd_calls = 0;
  h_mixed = 0;
  Dev dev;
  if (device_globals(&dev) != ST_OK) return;
  unsigned long long z[kNumCounters] = {};
  cudaDeviceSynchronize();
  cudaMemcpy(dev.counters, z, sizeof(z), cudaMemcpyHostToDevice);
}

st_status st_check_status(void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  st_status st = cuda_check(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  if (st != ST_OK) return st;
  Dev dev;
  if ((st = device_globals(&dev)) != ST_OK) return st;
  unsigned s = 0, z = 0;
  if ((st = cuda_check(cudaMemcpy(&s, dev.status, sizeof(s), cudaMemcpyDeviceToHost), "read status")) != ST_OK)
    return st;
  if (s & (kStatusTimeout | kStatusLayout)) {
    cudaMemcpy(dev.status, &z, sizeof(z), cudaMemcpyHostToDevice);
    if (s & kStatusLayout) return fail(ST_ERR_CUDA, "a kernel found its shared memory misaligned and did nothing");
    return fail(ST_ERR_TIMEOUT, "a kernel's bounded wait ran out");
  }
  return ST_OK;
}

}  // extern "C"
