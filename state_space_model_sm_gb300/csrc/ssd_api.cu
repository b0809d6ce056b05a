// C ABI of libssd (declared in include/ssd.h): argument checks, workspace
// carving and dispatch to the kernel families.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "ssd_internal.h"

namespace ssd {

__device__ int g_device_status = 0;

namespace {

std::atomic<int> g_check_finite{0};

// Records SSD_ERR_NONFINITE in the status word when any of n values is NaN or
// Inf (an earlier status is kept).  bf16 values are checked on their exponent
// field directly.
__global__ void k_check_finite(const void* p, int64_t n, int is_bf16, int* status) {
  bool bad = false;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (is_bf16) {
    const uint16_t* v = static_cast<const uint16_t*>(p);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
      bad |= (v[i] & 0x7F80u) == 0x7F80u;
  } else {
    const float* v = static_cast<const float*>(p);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
      bad |= !isfinite(v[i]);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
    atomicCAS(status, 0, (int)SSD_ERR_NONFINITE);
}

}  // namespace

bool check_finite_enabled() { return g_check_finite.load(std::memory_order_relaxed) != 0; }

// ------------------------------------------------------ launch-config table
namespace {
struct ScanEntry {
  int B, T, H, P, N, G, L;
  ssd_scan_config cfg;
};
constexpr int kMaxScanEntries = 64;
ScanEntry g_scan_table[kMaxScanEntries];
int g_scan_entries = 0;
std::mutex g_scan_mu;

// (entries hold the caller's shape; d may be the tensor-core path's view)
bool same_shape(const ScanEntry& e, const Dims& d) {
  return e.B == d.B && e.T == d.T && e.H == (d.H >> d.hs) && e.P == (d.P << d.hs) &&
         e.N == d.N && e.G == d.G && e.L == d.L;
}

// The built-in rule, a list-scheduling model of the launch: CTAs in grid
// order (every CTA of the heavier row tile first) each go to the SM that
// frees first, one at a time; a CTA costs its heads' 64-column operand
// uses (column panels + 4 per head) plus 6 for its prologue (the tile's rows
// and C.B^T).  The pair of head-block counts (divisors of the heads per
// group, at most 32) with the shortest modelled launch wins, fewer CTAs on a
// tie.  152 SMs: the GPU the tables were made on.  The model ranked the
// measured layer-shape pairs in their measured order.  For dC / dB, more than
// one block per tile also costs the tail's pass over the head-block partials
// (each row's slots read, the sum written, for both gradients), converted at
// the HBM copy rate into the same unit (one operand use ~ 1100 cycles at
// 2.07 GHz).
constexpr int kRuleSms = 152;
constexpr double kUseSeconds = 1100.0 / 2.07e9, kHbmBytesPerSecond = 6.8e12;

double model_makespan(int64_t n_heavy, double c_heavy, int64_t n_light, double c_light) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
  for (int i = 0; i < kRuleSms; ++i) sm.push(0.0);
  double end = 0.0;
  auto place = [&](int64_t n, double cost) {
    for (int64_t k = 0; k < n; ++k) {
      const double t = sm.top() + cost;
      sm.pop();
      sm.push(t);
      if (t > end) end = t;
    }
  };
  place(n_heavy, c_heavy);
  place(n_light, c_light);
  return end;
}

HeadBlocks rule_blocks_uncached(const Dims& d, bool partials) {
  const int hpg = d.H / d.G;
  const int64_t units = (int64_t)d.B * d.nc * d.G;  // per row tile
  std::vector<int> div;
  for (int nb = 1; nb <= hpg && nb <= 32; ++nb)
    if (hpg % nb == 0) div.push_back(nb);
  const double o = 6.0, heavy_uses = d.L / 64 + 4, light_uses = 2 + 4;
  const double row_bytes = 2.0 * d.B * d.T * d.G * d.N * 4.0;  // dB and dC, one slot
  auto tail = [&](int nmax) {
    return partials && nmax > 1 ? row_bytes * (nmax + 1) / kHbmBytesPerSecond / kUseSeconds
                                : 0.0;
  };
  HeadBlocks best{div[0], div[0]};
  double best_t = 1e300;
  int64_t best_n = 0;
  if (d.L <= 128) {  // one row tile
    for (const int nb : div) {
      const double t = model_makespan(units * nb, (hpg / nb) * light_uses + o, 0, 0.0) + tail(nb);
      if (t < best_t - 1e-9 || (t < best_t + 1e-9 && units * nb < best_n)) {
        best_t = t;
        best_n = units * nb;
        best = HeadBlocks{nb, nb};
      }
    }
    return best;
  }
  for (const int nh : div)
    for (const int nl : div) {
      const double t = model_makespan(units * nh, (hpg / nh) * heavy_uses + o, units * nl,
                                      (hpg / nl) * light_uses + o) +
                       tail(nh > nl ? nh : nl);
      const int64_t n = units * (nh + nl);
      if (t < best_t - 1e-9 || (t < best_t + 1e-9 && n < best_n)) {
        best_t = t;
        best_n = n;
        best = HeadBlocks{nh, nl};
      }
    }
  return best;
}

// the rule's choice per shape, computed once (the model takes milliseconds
// at long-context shapes)
struct RuleEntry {
  int B, T, H, P, N, G, L;
  HeadBlocks scan, bc;  // chunk_scan; dC / dB (with the tail's partial sums)
};
constexpr int kMaxRuleEntries = 64;
RuleEntry g_rule_cache[kMaxRuleEntries];
int g_rule_entries = 0, g_rule_next = 0;
std::mutex g_rule_mu;

HeadBlocks rule_blocks(const Dims& d, bool bc) {
  {
    std::lock_guard<std::mutex> lk(g_rule_mu);
    for (int i = 0; i < g_rule_entries; ++i) {
      const RuleEntry& e = g_rule_cache[i];
      if (e.B == d.B && e.T == d.T && e.H == d.H && e.P == d.P && e.N == d.N && e.G == d.G &&
          e.L == d.L)
        return bc ? e.bc : e.scan;
    }
  }
  const HeadBlocks sc = rule_blocks_uncached(d, false), b = rule_blocks_uncached(d, true);
  std::lock_guard<std::mutex> lk(g_rule_mu);
  const int i = g_rule_entries < kMaxRuleEntries ? g_rule_entries++ : (g_rule_next++ % kMaxRuleEntries);
  g_rule_cache[i] = RuleEntry{d.B, d.T, d.H, d.P, d.N, d.G, d.L, sc, b};
  return bc ? b : sc;
}

bool scan_lookup(const Dims& d, ssd_scan_config* out) {
  std::lock_guard<std::mutex> lk(g_scan_mu);
  for (int i = 0; i < g_scan_entries; ++i)
    if (same_shape(g_scan_table[i], d)) {
      *out = g_scan_table[i].cfg;
      return true;
    }
  return false;
}
}  // namespace

// a table field > 0 overrides the rule's count for that tile
HeadBlocks pick_blocks(const Dims& d, bool bc, int heavy, int light) {
  HeadBlocks hb = rule_blocks(d, bc);
  if (heavy > 0) hb.heavy = heavy;
  if (light > 0) hb.light = light;
  if (d.L <= 128) hb.light = hb.heavy;  // one row tile
  return hb;
}

HeadBlocks tc_scan_blocks(const Dims& d0) {
  const Dims d = tc_dims(d0);  // blocks of 64-wide head parts
  ssd_scan_config c{};
  if (!scan_lookup(d, &c)) return pick_blocks(d, false, 0, 0);
  return pick_blocks(d, false, c.scan_head_blocks, c.scan_head_blocks_light);
}

HeadBlocks tc_bwd_blocks(const Dims& d0) {
  const Dims d = tc_dims(d0);
  ssd_scan_config c{};
  if (!scan_lookup(d, &c)) return pick_blocks(d, true, 0, 0);
  return pick_blocks(d, true, c.bc_head_blocks, c.bc_head_blocks_light);
}

cudaError_t launch_check_finite(const void* p, int64_t n, bool is_bf16, cudaStream_t s) {
  if (!p || n <= 0) return cudaSuccess;
  int* status = device_status_ptr();
  if (!status) return cudaErrorUnknown;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + 255) / 256;
  const int grid = (int)(want < 4LL * sms ? want : 4LL * sms);
  SSD_LAUNCH("k_check_finite", s, k_check_finite<<<grid, 256, 0, s>>>(p, n, is_bf16, status));
  return cudaGetLastError();
}

int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

namespace {

thread_local int t_last_path = 0;

constexpr size_t kAlign = 256;

bool valid_dtype(int32_t v) { return v == SSD_F32 || v == SSD_BF16; }

int make_dims(const ssd_shape* s, Dims* d) {
  if (!s) return SSD_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seqlen < 1 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
      s->ngroups < 1 || s->chunk_size < 1)
    return SSD_ERR_INVALID_ARG;
  if (s->nheads % s->ngroups != 0) return SSD_ERR_INVALID_ARG;
  if (!valid_dtype(s->in_dtype) || !valid_dtype(s->out_dtype)) return SSD_ERR_INVALID_ARG;
  if (s->chunk_size > 256) return SSD_ERR_UNSUPPORTED;
  if (s->headdim * s->dstate > 16384) return SSD_ERR_UNSUPPORTED;
  // Keep every tensor's element count within int64 and every per-dimension
  // index within int32 (the kernels index a dimension with int).
  const int64_t lim = (int64_t)1 << 31;
  if (s->batch >= lim || s->seqlen >= lim || s->nheads >= 65536 || s->batch >= 65536)
    return SSD_ERR_UNSUPPORTED;
  const int64_t nc = (s->seqlen + s->chunk_size - 1) / s->chunk_size;
  if (nc >= lim) return SSD_ERR_UNSUPPORTED;
  d->B = (int)s->batch;
  d->T = (int)s->seqlen;
  d->H = (int)s->nheads;
  d->P = (int)s->headdim;
  d->N = (int)s->dstate;
  d->G = (int)s->ngroups;
  d->L = (int)s->chunk_size;
  d->nc = (int)nc;
  d->in_bf16 = s->in_dtype == SSD_BF16;
  d->out_bf16 = s->out_dtype == SSD_BF16;
  return SSD_OK;
}

struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  }
};

struct FwdOffsets {
  size_t delta, acs, S, Hprev, CB, seg, total;
};

// two-level state passing scratch: E and In, (B, K, H, P, N) floats each
size_t seg_bytes(const Dims& d) {
  return 2 * (size_t)d.B * seg_max_segments(d) * d.H * d.P * d.N * sizeof(float);
}

FwdOffsets fwd_offsets(const Dims& d) {
  Carver c;
  const size_t vec = (size_t)d.B * d.H * d.nc * d.L * sizeof(float);
  const size_t st = (size_t)d.B * d.nc * d.H * d.P * d.N * sizeof(float);
  FwdOffsets o;
  o.delta = c.take(vec);
  o.acs = c.take(vec);
  o.S = c.take(st);
  o.Hprev = c.take(st);
  o.CB = c.take((size_t)d.B * d.nc * d.G * d.L * d.L * sizeof(float));
  o.seg = c.take(seg_bytes(d));
  o.total = c.off;
  return o;
}

struct BwdOffsets {
  FwdOffsets f;
  size_t dHs, dS, dlast, dyx, qrow, ddir, ycs, dBh, dCh, part, total;
};

BwdOffsets bwd_offsets(const Dims& d) {
  BwdOffsets o;
  o.f = fwd_offsets(d);
  Carver c;
  c.off = o.f.total;
  const size_t vec = (size_t)d.B * d.H * d.nc * d.L * sizeof(float);
  const size_t st = (size_t)d.B * d.nc * d.H * d.P * d.N * sizeof(float);
  const size_t ph = (size_t)d.B * d.T * d.H * d.N * sizeof(float);
  o.dHs = c.take(st);
  o.dS = c.take(st);
  o.dlast = c.take((size_t)d.B * d.H * d.nc * 16 * sizeof(float));  // <= 16 partials each
  o.dyx = c.take((size_t)d.B * d.nc * d.H * d.L * d.L * sizeof(float));
  o.qrow = c.take(vec);
  o.ddir = c.take(vec);
  o.ycs = c.take(vec);
  o.dBh = c.take(ph);
  o.dCh = c.take(ph);
  o.part = c.take((size_t)d.B * d.H * d.nc * 3 * sizeof(float));
  o.total = c.off;
  return o;
}

struct TcBwdOffsets {
  size_t delta, acs, S, Himg, dHs, dSimg, dlast, rowsum, colsum, ycs, qrow, ddir, ddiag, dBp,
      dCp, part, done, seg, total;
};

TcBwdOffsets tc_bwd_offsets(const Dims& d, int nblk) {
  Carver c;
  const size_t vec = (size_t)d.B * d.H * d.nc * d.L * sizeof(float);
  const size_t st = (size_t)d.B * d.nc * d.H * d.P * d.N * sizeof(float);
  const size_t bp = (size_t)d.B * d.T * d.G * nblk * d.N * sizeof(float);
  TcBwdOffsets o;
  o.delta = c.take(vec);
  o.acs = c.take(vec);
  o.S = c.take(st);
  o.Himg = c.take(st);
  o.dHs = c.take(st);
  o.dSimg = c.take(st);
  o.dlast = c.take((size_t)d.B * d.H * d.nc * 64 * sizeof(float));  // <= 64 partials each
  o.rowsum = c.take(vec);
  o.colsum = c.take(vec);
  o.ycs = c.take(vec);
  o.qrow = c.take(vec);
  o.ddir = c.take(vec);
  o.ddiag = c.take(vec);
  o.dBp = c.take(bp);
  o.dCp = c.take(bp);
  o.part = c.take((size_t)d.B * d.H * d.nc * 3 * sizeof(float));
  o.done = c.take(sizeof(int));
  o.seg = c.take(seg_bytes(d));
  o.total = c.off;
  return o;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// SSD_FORCE_SIMT=1 in the environment keeps every call on the generic kernels.
bool force_simt() {
  const char* v = std::getenv("SSD_FORCE_SIMT");
  return v && v[0] == '1';
}

int check_fwd_ptrs(const Dims& d, const FwdArgs& a) {
  if (!a.x || !a.dt || !a.A || !a.B || !a.C) return SSD_ERR_INVALID_ARG;
  const size_t in = d.in_bf16 ? 2 : 4;
  if (!aligned(a.x, in) || !aligned(a.dt, in) || !aligned(a.B, in) || !aligned(a.C, in))
    return SSD_ERR_INVALID_ARG;
  const float* fp[] = {a.dt_bias, a.A, a.D, a.init, a.final_state};
  for (const float* p : fp)
    if (p && !aligned(p, 4)) return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

size_t seg_bytes_of(const FwdOffsets& o) { return o.total - o.seg; }

FwdWs carve_fwd(char* base, const FwdOffsets& o) {
  FwdWs w;
  w.delta = reinterpret_cast<float*>(base + o.delta);
  w.acs = reinterpret_cast<float*>(base + o.acs);
  w.S = reinterpret_cast<float*>(base + o.S);
  w.Hprev = reinterpret_cast<float*>(base + o.Hprev);
  w.CB = reinterpret_cast<float*>(base + o.CB);
  w.Himg = nullptr;
  w.seg = seg_bytes_of(o) ? reinterpret_cast<float*>(base + o.seg) : nullptr;
  return w;
}

// The opt-in scan of every gradient ssd_bwd wrote.
cudaError_t check_bwd_outputs(const Dims& d, const BwdArgs& a, cudaStream_t s) {
  if (!check_finite_enabled()) return cudaSuccess;
  const int64_t tok = (int64_t)d.B * d.T;
  const struct { const float* p; int64_t n; } outs[] = {
      {a.dx, tok * d.H * d.P}, {a.ddt, tok * d.H},       {a.dA, d.H},
      {a.dB, tok * d.G * d.N}, {a.dC, tok * d.G * d.N},   {a.dD, d.H},
      {a.ddt_bias, d.H},       {a.dinit, (int64_t)d.B * d.H * d.P * d.N}};
  for (const auto& o : outs) {
    const cudaError_t e = launch_check_finite(o.p, o.n, false, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_fwd_workspace_size(const ssd_shape* shape) {
  Dims d;
  if (make_dims(shape, &d) != SSD_OK) return 0;
  return fwd_offsets(d).total;
}

size_t ssd_bwd_workspace_size(const ssd_shape* shape) {
  Dims d;
  if (make_dims(shape, &d) != SSD_OK) return 0;
  size_t total = bwd_offsets(d).total;
  if (tc_forward_supported(d)) {
    const size_t t = tc_bwd_offsets(tc_dims(d), tc_bwd_blocks(d).max()).total;
    if (t > total) total = t;
  }
  return total;
}

int ssd_fwd_workspace_layout(const ssd_shape* shape, ssd_fwd_layout* out) {
  Dims d;
  const int st = make_dims(shape, &d);
  if (st != SSD_OK) return st;
  if (!out) return SSD_ERR_INVALID_ARG;
  const FwdOffsets o = fwd_offsets(d);
  out->delta = o.delta;
  out->dA_cumsum = o.acs;
  out->states = o.S;
  out->hprev = o.Hprev;
  out->total = o.total;
  return SSD_OK;
}

int ssd_fwd(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* init_states, void* y, float* final_states, void* workspace,
            size_t workspace_bytes, void* stream) {
  Dims d;
  int st = make_dims(shape, &d);
  if (st != SSD_OK) return st;
  FwdArgs a{x, dt, dt_bias, A, B, C, D, init_states, y, final_states};
  st = check_fwd_ptrs(d, a);
  if (st != SSD_OK) return st;
  if (!y || !aligned(y, d.out_bf16 ? 2 : 4)) return SSD_ERR_INVALID_ARG;
  const FwdOffsets o = fwd_offsets(d);
  if (!workspace || workspace_bytes < o.total || !aligned(workspace, kAlign))
    return SSD_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  FwdWs w = carve_fwd(static_cast<char*>(workspace), o);
  const bool tc = !force_simt() && tc_forward_supported(d) && aligned(x, 16) && aligned(B, 16) &&
                  aligned(C, 16) && aligned(y, 16) && aligned(init_states, 16) &&
                  aligned(final_states, 16);
  if (tc) {
    // the tensor-core kernels read the states as split-bf16 images, written in
    // place of the fp32 states (same bytes; see ssd_fwd_layout)
    w.Himg = w.Hprev;
    w.Hprev = nullptr;
  }
  t_last_path = tc ? 1 : 0;
  cudaError_t e = tc ? tc_forward(d, a, w, s) : simt_forward(d, a, w, s);
  if (e == cudaSuccess && check_finite_enabled()) {
    const int64_t ny = (int64_t)d.B * d.T * d.H * d.P;
    e = launch_check_finite(y, ny, d.out_bf16, s);
    if (e == cudaSuccess)
      e = launch_check_finite(final_states, (int64_t)d.B * d.H * d.P * d.N, false, s);
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_bwd(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* init_states, const void* dy, const float* dfinal_states, float* dx,
            float* ddt, float* dA, float* dB, float* dC, float* dD, float* ddt_bias,
            float* dinit_states, void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int st = make_dims(shape, &d);
  if (st != SSD_OK) return st;
  BwdArgs a;
  a.f = FwdArgs{x, dt, dt_bias, A, B, C, D, init_states, nullptr, nullptr};
  st = check_fwd_ptrs(d, a.f);
  if (st != SSD_OK) return st;
  a.dy = dy;
  a.dfinal = dfinal_states;
  a.dx = dx;
  a.ddt = ddt;
  a.dA = dA;
  a.dB = dB;
  a.dC = dC;
  a.dD = dD;
  a.ddt_bias = ddt_bias;
  a.dinit = dinit_states;
  if (!dy || !dx || !ddt || !dA || !dB || !dC) return SSD_ERR_INVALID_ARG;
  if (!aligned(dy, d.in_bf16 ? 2 : 4)) return SSD_ERR_INVALID_ARG;
  const float* fp[] = {dfinal_states, dx, ddt, dA, dB, dC, dD, ddt_bias, dinit_states};
  for (const float* p : fp)
    if (p && !aligned(p, 4)) return SSD_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  const bool tc = !force_simt() && tc_forward_supported(d) && aligned(x, 16) && aligned(B, 16) &&
                  aligned(C, 16) && aligned(dy, 16) && aligned(dx, 16) && aligned(dB, 16) &&
                  aligned(dC, 16) && aligned(init_states, 16) && aligned(dfinal_states, 16) &&
                  aligned(dinit_states, 16);
  if (tc) {
    const HeadBlocks nb = tc_bwd_blocks(d);  // once: the layout and the launch must agree
    // sized for the 64-wide head parts (the per-part row vectors of ddA)
    const TcBwdOffsets o = tc_bwd_offsets(tc_dims(d), nb.max());
    if (!workspace || workspace_bytes < o.total || !aligned(workspace, kAlign))
      return SSD_ERR_WORKSPACE;
    TcBwdWs w;
    w.delta = reinterpret_cast<float*>(base + o.delta);
    w.acs = reinterpret_cast<float*>(base + o.acs);
    w.S = reinterpret_cast<float*>(base + o.S);
    w.Himg = base + o.Himg;
    w.dHs = reinterpret_cast<float*>(base + o.dHs);
    w.dSimg = base + o.dSimg;
    w.dlast = reinterpret_cast<float*>(base + o.dlast);
    w.rowsum = reinterpret_cast<float*>(base + o.rowsum);
    w.colsum = reinterpret_cast<float*>(base + o.colsum);
    w.ycs = reinterpret_cast<float*>(base + o.ycs);
    w.qrow = reinterpret_cast<float*>(base + o.qrow);
    w.ddir = reinterpret_cast<float*>(base + o.ddir);
    w.ddiag = reinterpret_cast<float*>(base + o.ddiag);
    w.dBp = reinterpret_cast<float*>(base + o.dBp);
    w.dCp = reinterpret_cast<float*>(base + o.dCp);
    w.part = reinterpret_cast<float*>(base + o.part);
    w.done = reinterpret_cast<int*>(base + o.done);
    w.seg = o.total > o.seg ? reinterpret_cast<float*>(base + o.seg) : nullptr;
    w.nb = nb;
    t_last_path = 1;
    if (tc_backward(d, a, w, s) != cudaSuccess) return SSD_ERR_CUDA;
    return check_bwd_outputs(d, a, s) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  const BwdOffsets o = bwd_offsets(d);
  if (!workspace || workspace_bytes < o.total || !aligned(workspace, kAlign))
    return SSD_ERR_WORKSPACE;
  BwdWs w;
  w.f = carve_fwd(base, o.f);
  w.f.Himg = nullptr;
  w.dHs = reinterpret_cast<float*>(base + o.dHs);
  w.dS = reinterpret_cast<float*>(base + o.dS);
  w.dlast = reinterpret_cast<float*>(base + o.dlast);
  w.dyx = reinterpret_cast<float*>(base + o.dyx);
  w.qrow = reinterpret_cast<float*>(base + o.qrow);
  w.ddir = reinterpret_cast<float*>(base + o.ddir);
  w.ycs = reinterpret_cast<float*>(base + o.ycs);
  w.dBh = reinterpret_cast<float*>(base + o.dBh);
  w.dCh = reinterpret_cast<float*>(base + o.dCh);
  w.part = reinterpret_cast<float*>(base + o.part);
  t_last_path = 0;
  if (simt_backward(d, a, w, s) != cudaSuccess) return SSD_ERR_CUDA;
  return check_bwd_outputs(d, a, s) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_fwd_final_state(const ssd_shape* shape, const void* x, const void* dt,
                        const float* dt_bias, const float* A, const void* B,
                        const float* init_states, float* final_states, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Dims d;
  int st = make_dims(shape, &d);
  if (st != SSD_OK) return st;
  if (!x || !dt || !A || !B || !final_states) return SSD_ERR_INVALID_ARG;
  const size_t in = d.in_bf16 ? 2 : 4;
  if (!aligned(x, in) || !aligned(dt, in) || !aligned(B, in)) return SSD_ERR_INVALID_ARG;
  const float* fp[] = {dt_bias, A, init_states, final_states};
  for (const float* p : fp)
    if (p && !aligned(p, 4)) return SSD_ERR_INVALID_ARG;
  const FwdOffsets o = fwd_offsets(d);
  if (!workspace || workspace_bytes < o.total || !aligned(workspace, kAlign))
    return SSD_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const FwdArgs a{x, dt, dt_bias, A, B, nullptr, nullptr, init_states, nullptr, final_states};
  FwdWs w = carve_fwd(static_cast<char*>(workspace), o);
  const bool tc = !force_simt() && tc_forward_supported(d) && aligned(x, 16) && aligned(B, 16) &&
                  aligned(init_states, 16) && aligned(final_states, 16);
  t_last_path = tc ? 1 : 0;
  if (tc) {
    w.Himg = w.Hprev;  // the state images take the fp32 states' place, as in ssd_fwd
    w.Hprev = nullptr;
    return tc_front_final(d, a, w, s) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  simt_front(d, a, w, s);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_bwd_dinit(const ssd_shape* shape, const void* dt, const float* dt_bias, const float* A,
                  const void* C, const void* dy, const float* dfinal_states,
                  float* dinit_states, void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int st = make_dims(shape, &d);
  if (st != SSD_OK) return st;
  if (!dt || !A || !C || !dy || !dinit_states) return SSD_ERR_INVALID_ARG;
  const size_t in = d.in_bf16 ? 2 : 4;
  if (!aligned(dt, in) || !aligned(C, in) || !aligned(dy, in)) return SSD_ERR_INVALID_ARG;
  const float* fp[] = {dt_bias, A, dfinal_states, dinit_states};
  for (const float* p : fp)
    if (p && !aligned(p, 4)) return SSD_ERR_INVALID_ARG;
  const FwdOffsets o = fwd_offsets(d);
  if (!workspace || workspace_bytes < o.total || !aligned(workspace, kAlign))
    return SSD_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const FwdArgs a{nullptr, dt, dt_bias, A, nullptr, C, nullptr, nullptr, nullptr, nullptr};
  const FwdWs w = carve_fwd(static_cast<char*>(workspace), o);
  float* dHs = w.S;  // the chunk-state slot holds dH^scan here
  const bool tc = !force_simt() && tc_forward_supported(d) && aligned(C, 16) && aligned(dy, 16);
  t_last_path = tc ? 1 : 0;
  simt_cumsum(d, a, w, s);
  if (tc) {
    if (tc_dstates(d, dy, C, w.delta, w.acs, dHs, s) != cudaSuccess) return SSD_ERR_CUDA;
  } else {
    simt_dstates(d, dy, C, w.delta, w.acs, dHs, s);
  }
  cp_dinit_chain(d, dHs, w.acs, dfinal_states, dinit_states, s);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSD_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return SSD_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
    return SSD_ERR_CUDA;
  return v;
}

int ssd_last_path(void) { return t_last_path; }

int ssd_set_check_finite(int enable) { return g_check_finite.exchange(enable ? 1 : 0); }

int ssd_scan_set_config(const ssd_shape* shape, const ssd_scan_config* config) {
  Dims d;
  if (make_dims(shape, &d) != SSD_OK) return SSD_ERR_INVALID_ARG;
  if (config) {
    const int hpg = tc_dims(d).H / d.G;  // 64-wide head parts per group
    for (const int v : {config->scan_head_blocks, config->bc_head_blocks,
                         config->scan_head_blocks_light, config->bc_head_blocks_light})
      if (v < 0 || v > 32 || (v > 0 && hpg % v != 0)) return SSD_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_scan_mu);
  int i = 0;
  while (i < g_scan_entries && !same_shape(g_scan_table[i], d)) ++i;
  if (!config) {  // remove
    if (i < g_scan_entries) g_scan_table[i] = g_scan_table[--g_scan_entries];
    return SSD_OK;
  }
  if (i == g_scan_entries) {
    if (g_scan_entries == kMaxScanEntries) return SSD_ERR_UNSUPPORTED;
    ++g_scan_entries;
  }
  g_scan_table[i] = ScanEntry{d.B, d.T, d.H, d.P, d.N, d.G, d.L, *config};
  return SSD_OK;
}

int ssd_scan_get_config(const ssd_shape* shape, ssd_scan_config* out) {
  Dims d;
  if (!out || make_dims(shape, &d) != SSD_OK) return -SSD_ERR_INVALID_ARG;
  ssd_scan_config c{};
  const bool set = scan_lookup(d, &c);
  const HeadBlocks sc = tc_scan_blocks(d), bc = tc_bwd_blocks(d);
  out->scan_head_blocks = sc.heavy;
  out->scan_head_blocks_light = sc.light;
  out->bc_head_blocks = bc.heavy;
  out->bc_head_blocks_light = bc.light;
  return set ? 1 : 0;
}

const char* ssd_strerror(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument (shape, NULL pointer or alignment)";
    case SSD_ERR_UNSUPPORTED: return "shape outside what the kernels implement";
    case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSD_ERR_CUDA: return "CUDA runtime or launch error";
    case SSD_ERR_TIMEOUT: return "device-side bounded wait timed out";
    case SSD_ERR_NONFINITE: return "an output holds NaN or Inf";
    default: return "unknown status";
  }
}

}  // extern "C"
