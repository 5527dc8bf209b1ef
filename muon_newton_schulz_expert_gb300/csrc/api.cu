// C ABI of libmuon: argument checks, workspace layout, the order of the
// kernels of one Muon step, device status and tracing.
//
// Source of the step: "Training a 1T-Parameter MoE on EU public
// infrastructure with PyTorch and TorchTitan", section "FlexShard: Muon without
// communication" (one fp32 state per parameter; a few Newton-Schulz iterations
// on each whole matrix; whole-expert ownership, so no communication).
#include <math.h>

#include <cmath>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace muon {

__device__ unsigned g_muon_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_fail_allocs{0};   // injected allocation failures still pending

const char *kTraceNames[kTraceKinds] = {"momentum_bf16", "momentum_f32", "norm_partial", "norm_final",
                                        "transpose",     "scale",        "ns_syrk_tc",   "ns_poly_tc",
                                        "ns_axpy_tc",    "apply_bf16",   "apply_f32",    "gemm_f32",
                                        "copy",          "selftest_wait", "adamw",       "momentum_norm_bf16",
                                        "ns_axpy_apply_tc"};

struct TraceRec {
  int kind;
  cudaEvent_t start, stop;
};

struct Tracer {
  bool on = false;
  std::vector<TraceRec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t pending_start = nullptr;
} g_trace;

cudaEvent_t take_event() {
  if (!g_trace.pool.empty()) {
    cudaEvent_t e = g_trace.pool.back();
    g_trace.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// ------------------------------------------------------------ internal services
void trace_before(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_trace.on) return;
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, s) == cudaSuccess) g_trace.pending_start = e;
  (void)kind;
}

int trace_after(int kind, cudaStream_t s) {
  cudaError_t err = cudaGetLastError();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_trace.on && g_trace.pending_start) {
      cudaEvent_t e = take_event();
      if (e && cudaEventRecord(e, s) == cudaSuccess) g_trace.recs.push_back({kind, g_trace.pending_start, e});
      g_trace.pending_start = nullptr;
    }
  }
  return err == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

unsigned *device_error_word() {
  int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_muon_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<unsigned *>(p);
  }
  return g_err_ptr[d];
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }

int num_sms() {
  int d = current_device();
  if (d < 0) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) v = 148;
    g_sms[d] = v;
  }
  return g_sms[d];
}

cudaError_t alloc_async(void **ptr, size_t bytes, cudaStream_t s) {
  int pending = g_fail_allocs.load();
  while (pending > 0)
    if (g_fail_allocs.compare_exchange_weak(pending, pending - 1)) return cudaErrorMemoryAllocation;
  return cudaMallocAsync(ptr, bytes, s);
}

namespace {

// Workspace of one Newton-Schulz call on [batch][mm][nn] (mm <= nn), in order:
// two X buffers, the low half of X (tensor-core path only, one byte per
// element), A, B (mm x mm each), norm partials, 1/(||X||+eps) and its square.  Every region starts on
// a 256-byte boundary and is followed by kGapBytes that no kernel writes, so
// that a write past a region's end lands in a gap a test can inspect rather
// than in the next region.
struct Workspace {
  void *x1, *x2, *lo, *a, *b;
  float *partial, *inv, *inv2;
};

constexpr size_t kGapBytes = 256;

inline size_t region(size_t bytes) { return align256(bytes) + kGapBytes; }

// X's low half, one byte per element, rows padded to 16 bytes (TMA strides):
// room for either storage orientation
inline size_t pitch16(int64_t cols) { return (size_t)((cols + 15) & ~int64_t(15)); }
inline size_t lo_bytes(int64_t batch, int64_t mm, int64_t nn) {
  return (size_t)batch * std::max((size_t)mm * pitch16(nn), (size_t)nn * pitch16(mm));
}

size_t ws_bytes(int64_t batch, int64_t mm, int64_t nn, size_t elem) {
  const size_t xs = region((size_t)batch * mm * nn * elem);
  const size_t los = elem == 2 ? region(lo_bytes(batch, mm, nn)) : 0;
  const size_t as = region((size_t)batch * mm * mm * elem);
  const size_t fl = region((size_t)batch * norm_partials() * sizeof(float)) + 2 * region((size_t)batch * sizeof(float));
  return 2 * xs + los + 2 * as + fl;
}

Workspace carve(void *base, int64_t batch, int64_t mm, int64_t nn, size_t elem) {
  uint8_t *p = static_cast<uint8_t *>(base);
  Workspace w{};
  const size_t xs = region((size_t)batch * mm * nn * elem);
  const size_t as = region((size_t)batch * mm * mm * elem);
  w.x1 = p;
  p += xs;
  w.x2 = p;
  p += xs;
  if (elem == 2) {
    w.lo = p;
    p += region(lo_bytes(batch, mm, nn));
  }
  w.a = p;
  p += as;
  w.b = p;
  p += as;
  w.partial = reinterpret_cast<float *>(p);
  p += region((size_t)batch * norm_partials() * sizeof(float));
  w.inv = reinterpret_cast<float *>(p);
  p += region((size_t)batch * sizeof(float));
  w.inv2 = reinterpret_cast<float *>(p);
  return w;
}

// ncoeff: how many floats `coeffs` holds (3, or 3 * steps for a schedule)
int check_ns_args(const void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs, float eps,
                  int64_t ncoeff = 3) {
  if (batch < 0 || m < 1 || n < 1 || steps < 0 || !coeffs) return MUON_ERR_INVALID_ARG;
  if (steps > 1000) return MUON_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !isfinite(eps)) return MUON_ERR_INVALID_ARG;
  for (int64_t i = 0; i < ncoeff; ++i)
    if (!isfinite(coeffs[i])) return MUON_ERR_INVALID_ARG;
  if (batch > 0 && !X) return MUON_ERR_INVALID_ARG;
  if (m > (1 << 20) || n > (1 << 20) || batch > (int64_t(1) << 31)) return MUON_ERR_UNSUPPORTED;
  return MUON_OK;
}

#define MUON_TRY(expr)          \
  do {                          \
    int _st = (expr);           \
    if (_st != MUON_OK) return _st; \
  } while (0)

int copy_async(void *dst, const void *src, size_t bytes, cudaStream_t s) {
  trace_before(kTraceCopy, s);
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  int st = trace_after(kTraceCopy, s);
  return e == cudaSuccess ? st : MUON_ERR_CUDA;
}

// Storage plan of the tensor-core iteration.  What an iteration produces (A,
// B and X's high half) is stored in 16 bits, in one of two formats chosen per
// call by the matrix size:
//  - bf16, for m > kF16MaxRows: the computed values rounded to bf16, no
//    scaling;
//  - fp16 scaled by powers of two, for m <= kF16MaxRows, except the first
//    iteration's B, which stays bf16 because it meets the bf16 input u in one
//    tensor-core product (kind::f16 takes both operands in one format).  A
//    value v is stored as fp16(sigma v), sigma chosen from a bound on the
//    matrix's spectral norm, which bounds every entry: ||X_0|| <= ||X_0||_F
//    <= 1 after the normalisation, and per step ||A|| = ||X||^2, ||B|| <=
//    max |b l + c l^2| over l in [0, ||A||] and ||X'|| <= max |a x + b x^3 +
//    c x^5| over x in [0, ||X||] (the iteration acts on each singular value
//    by these scalar maps).  The largest entry is then held near 2^14 (fp16
//    reaches 65504), and the powers of two fold exactly into the constants
//    each epilogue already applies.
// Why two formats: fp16 keeps 11 significant bits against bf16's 8.  With
// bf16 storage the output's error is ~1% of its norm on large matrices, but
// small ones have few singular directions to average the rounding over, and
// up to m ~ 16 a third of random inputs exceed 2% (a CPU model of these
// rounding points: tests/test_rounding_model.py); with fp16 storage every size
// stays near the 0.2% of the final bf16 rounding.  On large batches, though,
// fp16 products draw more power than bf16 ones, and under the board's power
// cap that lowered the clock and the step's throughput by 3.5%.  Matrices up
// to kF16MaxRows rows are small enough for that not to matter.
constexpr int64_t kF16MaxRows = 256;

struct IterPlan {
  float syrk_mul;          // sigma_A / sigma_in^2
  float poly_b, poly_c;    // b sigma_B / sigma_A, c sigma_B / sigma_A^2
  float axpy_a, axpy_mul;  // a sigma_B, sigma_out / (sigma_in sigma_B)
  float lo_in, lo_out;     // the low half's power-of-two factors: read (1/S) and written (S)
  int tin;                 // format of X and B in this iteration's product
  int store;               // format of A, and of B and X' unless bf16 is required
};

// max |a x + b x^3 + c x^5| over x in [0, hi]: the ends and the stationary
// points, x^2 = t a root of 5c t^2 + 3b t + a
double max_abs_quintic(double a, double b, double c, double hi) {
  auto f = [&](double x) { return fabs(x * (a + x * x * (b + c * x * x))); };
  double best = f(hi);
  double roots[2];
  int nr = 0;
  if (c != 0.0) {
    const double disc = 9.0 * b * b - 20.0 * a * c;
    if (disc >= 0.0) {
      const double sq = sqrt(disc);
      roots[nr++] = (-3.0 * b + sq) / (10.0 * c);
      roots[nr++] = (-3.0 * b - sq) / (10.0 * c);
    }
  } else if (b != 0.0) {
    roots[nr++] = -a / (3.0 * b);
  }
  for (int i = 0; i < nr; ++i)
    if (roots[i] > 0.0 && roots[i] < hi * hi) best = std::max(best, f(sqrt(roots[i])));
  return best;
}

// max |b l + c l^2| over l in [0, hi]
double max_abs_quad(double b, double c, double hi) {
  auto f = [&](double l) { return fabs(l * (b + c * l)); };
  double best = f(hi);
  if (c != 0.0) {
    const double l = -b / (2.0 * c);
    if (l > 0.0 && l < hi) best = std::max(best, f(l));
  }
  return best;
}

// exponent e of the power of two 2^e that puts `bound` (with 1% to spare)
// at or below 2^14; false when no such e within [-40, 40] exists
bool storage_exp(double bound, int *e) {
  if (!(bound > 1e-30)) {  // zero (or negligible) matrix: any scale stores it
    *e = 0;
    return true;
  }
  if (!std::isfinite(bound)) return false;
  const int k = 14 - (int)ceil(log2(bound * 1.01));
  if (k > 40) {
    *e = 40;
    return true;
  }
  if (k < -40) return false;
  *e = k;
  return true;
}

// X's low half, lo = x - hi with hi = x rounded to the storage format, is at
// most hi's rounding unit: |lo| <= 2^-8 |x| for bf16 (2^-11 for fp16), with
// x the stored value sigma X'.  It is kept in 8 bits as e5m2(lo * S) (five
// exponent bits, two of mantissa, finite up to 57344), S a power of two that
// puts the bound at 2^13 or below; e5m2's 31 binades below that keep every
// lo that matters (a CPU model of these rounding points puts the cost at
// <= 0.5% of the output's norm on the conditioning-stress inputs, against a
// 16-bit low half).
bool low_half_scale(double bound, int *e) {
  if (!(bound > 1e-30)) {
    *e = 0;
    return true;
  }
  if (!std::isfinite(bound)) return false;
  const int k = 13 - (int)ceil(log2(bound * 1.01));
  *e = std::max(-100, std::min(100, k));
  return true;
}

int plan_ns(int64_t mm, int steps, const float *cf, int cf_stride, std::vector<IterPlan> *plan) {
  plan->assign((size_t)steps, IterPlan{});
  const int store = mm <= kF16MaxRows ? kF16 : kBF16;
  double bx = 1.0;   // bound on ||X_k||
  int ex = 0;        // sigma_X of the current input (the first input carries s instead)
  int elo = 0;       // S of the current input's low half
  for (int it = 0; it < steps; ++it) {
    const double a = cf[(size_t)it * cf_stride], b = cf[(size_t)it * cf_stride + 1],
                 c = cf[(size_t)it * cf_stride + 2];
    const double bx_next = max_abs_quintic(a, b, c, bx);
    int ea = 0, eb = 0, eo = 0;
    if (store == kF16) {   // bf16 shares fp32's exponent range: no scaling
      const double ba = bx * bx, bb = max_abs_quad(b, c, ba);
      if (!storage_exp(ba, &ea)) return MUON_ERR_UNSUPPORTED;
      if (it > 0 && !storage_exp(bb, &eb)) return MUON_ERR_UNSUPPORTED;   // the first B is bf16
      if (it + 1 < steps && !storage_exp(bx_next, &eo)) return MUON_ERR_UNSUPPORTED;
    }
    int elo_out = 0;
    if (it + 1 < steps) {
      const double unit = store == kF16 ? ldexp(1.0, -11) : ldexp(1.0, -8);
      if (!low_half_scale(unit * ldexp(bx_next, eo), &elo_out)) return MUON_ERR_UNSUPPORTED;
    }
    const int ein = it == 0 ? 0 : ex;
    IterPlan &q = (*plan)[it];
    q.syrk_mul = (float)ldexp(1.0, ea - 2 * ein);
    q.poly_b = (float)ldexp(b, eb - ea);
    q.poly_c = (float)ldexp(c, eb - 2 * ea);
    q.axpy_a = (float)ldexp(a, eb);
    q.axpy_mul = (float)ldexp(1.0, eo - ein - eb);   // the last iteration stores the value itself
    q.lo_in = (float)ldexp(1.0, -elo);
    q.lo_out = (float)ldexp(1.0, elo_out);
    q.tin = it == 0 ? kBF16 : store;
    q.store = store;
    bx = bx_next;
    ex = eo;
    elo = elo_out;
  }
  return MUON_OK;
}

// Which iterates carry X's low half.  Rounding an iterate to 16 bits adds
// noise to every singular direction, and each later step multiplies small
// singular values by up to a (3.4445 for the quintic), so the low half
// matters most early: without it on the first step's output the
// conditioning-stress inputs reach 18% error.  The last step's input is the
// exception: its rounding passes through one step only (gain <= a), which
// costs at most 0.3% of the output's norm on those inputs (a CPU model of the
// rounding points, 1 to 6 steps), while dropping it saves 4 bytes per element
// of traffic: the low half's store in the second-to-last step and its load in
// the last.
inline bool writes_low_half(int it, int steps) { return it + 2 < steps; }
inline bool reads_low_half(int it, int steps) { return it > 0 && writes_low_half(it - 1, steps); }

// The tensor-core iteration on the canonical orientation.  `src0` holds X
// (bf16, mm x nn per matrix); the result (bf16) ends in `dst_final`, which may
// be src0 itself.  Intermediate iterates live in the workspace's two X
// buffers (fp16 high halves) and its low-half buffer.
// cf holds (a, b, c) for step it at cf + it * cf_stride (stride 0: one triple).
int ns_bf16_core(__nv_bfloat16 *src0, __nv_bfloat16 *dst_final, const Workspace &w, int64_t batch, int64_t mm,
                 int64_t nn, bool transposed, int steps, const float *cf, int cf_stride, float eps, cudaStream_t s) {
  const int64_t per = mm * nn;
  std::vector<IterPlan> plan;
  MUON_TRY(plan_ns(mm, steps, cf, cf_stride, &plan));
  MUON_TRY(launch_inv_norm_bf16(src0, batch, per, eps, w.partial, w.inv, w.inv2, s));
  if (steps == 0) return launch_scale_bf16(src0, dst_final, batch, per, w.inv, s);
  auto *lo = static_cast<uint8_t *>(w.lo);
  void *src = src0;
  for (int it = 0; it < steps; ++it) {
    const IterPlan &q = plan[it];
    const bool last = it == steps - 1;
    // the last iteration writes dst_final unless it would read and write the
    // same buffer (a single step on the caller's X): then it is copied over
    void *dst = last && src != dst_final ? static_cast<void *>(dst_final) : (src == w.x1 ? w.x2 : w.x1);
    MUON_TRY(ns_syrk(src, q.tin, w.a, q.store, batch, mm, nn, it == 0 ? w.inv2 : nullptr, q.syrk_mul, transposed, s));
    MUON_TRY(ns_poly(w.a, q.store, w.b, q.tin, batch, mm, q.poly_b, q.poly_c, s));
    // the first input is exactly bf16 (no low half); the result leaves as bf16
    MUON_TRY(ns_axpy(w.b, src, q.tin, reads_low_half(it, steps) ? lo : nullptr, q.lo_in, dst, last ? kBF16 : q.store,
                     writes_low_half(it, steps) ? lo : nullptr, q.lo_out, batch, mm, nn, q.axpy_a,
                     it == 0 ? w.inv : nullptr, q.axpy_mul, transposed, s));
    src = dst;
  }
  if (src != dst_final) MUON_TRY(copy_async(dst_final, src, (size_t)batch * per * 2, s));
  return MUON_OK;
}

int ns_f32_core(float *src0, float *final_dst, const Workspace &w, int64_t batch, int64_t mm, int64_t nn, int steps,
                const float *cf, int cf_stride, float eps, cudaStream_t s, float **result) {
  const int64_t per = mm * nn;
  MUON_TRY(launch_inv_norm_f32(src0, batch, per, eps, w.partial, w.inv, w.inv2, s));
  auto *x1 = static_cast<float *>(w.x1);
  auto *x2 = static_cast<float *>(w.x2);
  if (steps == 0) {
    *result = final_dst ? final_dst : src0;
    return launch_scale_f32(src0, *result, batch, per, w.inv, s);
  }
  auto *A = static_cast<float *>(w.a);
  auto *B = static_cast<float *>(w.b);
  float *src = src0;
  for (int it = 0; it < steps; ++it) {
    const bool last = it == steps - 1;
    float *dst = (src == x1) ? x2 : x1;
    if (last && final_dst && final_dst != src) dst = final_dst;
    const float *c = cf + (size_t)it * cf_stride;
    MUON_TRY(gemm_f32(0, src, nullptr, A, batch, mm, nn, 0.f, 0.f, 0.f, it == 0 ? w.inv2 : nullptr, s));
    MUON_TRY(gemm_f32(1, A, nullptr, B, batch, mm, mm, 0.f, c[1], c[2], nullptr, s));
    MUON_TRY(gemm_f32(2, B, src, dst, batch, mm, nn, c[0], 0.f, 0.f, it == 0 ? w.inv : nullptr, s));
    src = dst;
  }
  if (final_dst && src != final_dst) {
    MUON_TRY(copy_async(final_dst, src, (size_t)batch * per * 4, s));
    src = final_dst;
  }
  *result = src;
  return MUON_OK;
}

// Checked arguments; X in caller layout.  For m > n the iteration runs on X^T
// without moving data: the kernels read the stored matrix as the transpose of
// the canonical mm x nn one.
int ns_bf16_entry(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *cf, int cf_stride, float eps,
                  void *workspace, size_t workspace_bytes, cudaStream_t s) {
  if (batch == 0) return MUON_OK;
  if (m % 8 || n % 8 || !aligned16(X)) return MUON_ERR_UNSUPPORTED;
  std::vector<IterPlan> plan;
  MUON_TRY(plan_ns(std::min(m, n), steps, cf, cf_stride, &plan));
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MUON_ERR_INVALID_ARG;
  const int64_t mm = std::min(m, n), nn = std::max(m, n);
  if (workspace_bytes < ws_bytes(batch, mm, nn, 2)) return MUON_ERR_NO_MEMORY;
  if (!device_error_word()) return MUON_ERR_CUDA;
  Workspace w = carve(workspace, batch, mm, nn, 2);
  auto *x = static_cast<__nv_bfloat16 *>(X);
  return ns_bf16_core(x, x, w, batch, mm, nn, m > n, steps, cf, cf_stride, eps, s);
}

// Allocates the workspace stream-ordered on s around ns_bf16_entry.
int ns_bf16_alloc(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *cf, int cf_stride, float eps,
                  cudaStream_t s) {
  if (batch == 0) return MUON_OK;
  if (m % 8 || n % 8 || !aligned16(X)) return MUON_ERR_UNSUPPORTED;
  std::vector<IterPlan> plan;
  MUON_TRY(plan_ns(std::min(m, n), steps, cf, cf_stride, &plan));
  const size_t bytes = ws_bytes(batch, std::min(m, n), std::max(m, n), 2);
  void *ws = nullptr;
  if (alloc_async(&ws, bytes, s) != cudaSuccess || !ws) {
    cudaGetLastError();
    return MUON_ERR_NO_MEMORY;
  }
  int st = ns_bf16_entry(X, batch, m, n, steps, cf, cf_stride, eps, ws, bytes, s);
  cudaError_t fe = cudaFreeAsync(ws, s);
  if (st == MUON_OK && fe != cudaSuccess) st = MUON_ERR_CUDA;
  return st;
}

int ns_f32_alloc(float *X, int64_t batch, int64_t m, int64_t n, int steps, const float *cf, int cf_stride, float eps,
                 cudaStream_t s) {
  if (batch == 0) return MUON_OK;
  const size_t bytes = ws_bytes(batch, std::min(m, n), std::max(m, n), 4);
  void *ws = nullptr;
  if (alloc_async(&ws, bytes, s) != cudaSuccess || !ws) {
    cudaGetLastError();
    return MUON_ERR_NO_MEMORY;
  }
  const int64_t mm = std::min(m, n), nn = std::max(m, n);
  Workspace w = carve(ws, batch, mm, nn, 4);
  int st;
  float *res = nullptr;
  if (m <= n) {
    st = ns_f32_core(X, X, w, batch, mm, nn, steps, cf, cf_stride, eps, s, &res);
  } else {
    float *xt = static_cast<float *>(w.x1);
    st = launch_transpose_f32(X, xt, batch, m, n, s);
    if (st == MUON_OK) st = ns_f32_core(xt, nullptr, w, batch, mm, nn, steps, cf, cf_stride, eps, s, &res);
    if (st == MUON_OK) st = launch_transpose_f32(res, X, batch, mm, nn, s);
  }
  cudaError_t fe = cudaFreeAsync(ws, s);
  if (st == MUON_OK && fe != cudaSuccess) st = MUON_ERR_CUDA;
  return st;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" {

int muon_momentum_update(const void *grad, float *momentum, void *update_out, int64_t numel, float mu, int nesterov,
                         muon_stream_t stream) {
  if (numel < 0) return MUON_ERR_INVALID_ARG;
  if (numel == 0) return MUON_OK;
  if (!grad || !momentum || !update_out) return MUON_ERR_INVALID_ARG;
  return launch_momentum_bf16(static_cast<const __nv_bfloat16 *>(grad), momentum,
                              static_cast<__nv_bfloat16 *>(update_out), numel, mu, nesterov ? 1 : 0,
                              reinterpret_cast<cudaStream_t>(stream));
}

int muon_momentum_update_f32(const float *grad, float *momentum, float *update_out, int64_t numel, float mu,
                             int nesterov, muon_stream_t stream) {
  if (numel < 0) return MUON_ERR_INVALID_ARG;
  if (numel == 0) return MUON_OK;
  if (!grad || !momentum || !update_out) return MUON_ERR_INVALID_ARG;
  return launch_momentum_f32(grad, momentum, update_out, numel, mu, nesterov ? 1 : 0,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t muon_ns_workspace_bytes(int64_t batch, int64_t m, int64_t n) {
  if (batch <= 0 || m < 1 || n < 1) return 0;
  return ws_bytes(batch, std::min(m, n), std::max(m, n), 2);
}

size_t muon_ns_workspace_bytes_f32(int64_t batch, int64_t m, int64_t n) {
  if (batch <= 0 || m < 1 || n < 1) return 0;
  return ws_bytes(batch, std::min(m, n), std::max(m, n), 4);
}

}  // extern "C"

namespace muon {
int ns_precheck(const void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs, float eps) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps));
  if (batch > 0 && (m % 8 || n % 8 || !aligned16(X))) return MUON_ERR_UNSUPPORTED;
  std::vector<IterPlan> plan;
  return plan_ns(std::min(m, n), steps, coeffs, 0, &plan);
}
}  // namespace muon

extern "C" {

int muon_ns_batched_ws(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3], float eps,
                       void *workspace, size_t workspace_bytes, muon_stream_t stream) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps));
  const float cf[3] = {coeffs[0], coeffs[1], coeffs[2]};
  return ns_bf16_entry(X, batch, m, n, steps, cf, 0, eps, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int muon_ns_batched(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3], float eps,
                    muon_stream_t stream) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps));
  const float cf[3] = {coeffs[0], coeffs[1], coeffs[2]};
  return ns_bf16_alloc(X, batch, m, n, steps, cf, 0, eps, reinterpret_cast<cudaStream_t>(stream));
}

int muon_ns_batched_schedule(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs,
                             float eps, muon_stream_t stream) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps, 3 * (int64_t)steps));
  std::vector<float> cf(coeffs, coeffs + 3 * (size_t)steps);
  return ns_bf16_alloc(X, batch, m, n, steps, cf.data(), 3, eps, reinterpret_cast<cudaStream_t>(stream));
}

int muon_ns_batched_f32(float *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3], float eps,
                        muon_stream_t stream) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps));
  const float cf[3] = {coeffs[0], coeffs[1], coeffs[2]};
  return ns_f32_alloc(X, batch, m, n, steps, cf, 0, eps, reinterpret_cast<cudaStream_t>(stream));
}

int muon_ns_batched_schedule_f32(float *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs,
                                 float eps, muon_stream_t stream) {
  MUON_TRY(check_ns_args(X, batch, m, n, steps, coeffs, eps, 3 * (int64_t)steps));
  std::vector<float> cf(coeffs, coeffs + 3 * (size_t)steps);
  return ns_f32_alloc(X, batch, m, n, steps, cf.data(), 3, eps, reinterpret_cast<cudaStream_t>(stream));
}

float muon_default_scale(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 1) return 1.0f;
  return (float)sqrt(std::max(1.0, (double)rows / (double)cols));
}

static void update_constants(int64_t rows, int64_t cols, float lr, float wd, float scale, float *kw, float *ko) {
  const double sc = scale > 0.f ? (double)scale : sqrt(std::max(1.0, (double)rows / (double)cols));
  *kw = (float)(1.0 - (double)lr * (double)wd);
  *ko = (float)(-(double)lr * sc);
}

int muon_apply_update(void *param, const void *update, int64_t batch, int64_t rows, int64_t cols, float lr,
                      float weight_decay, float scale, muon_stream_t stream) {
  if (batch < 0 || rows < 0 || cols < 0) return MUON_ERR_INVALID_ARG;
  const int64_t numel = batch * rows * cols;
  if (numel == 0) return MUON_OK;
  if (!param || !update || !isfinite(lr) || !isfinite(weight_decay) || !isfinite(scale)) return MUON_ERR_INVALID_ARG;
  float kw, ko;
  update_constants(rows, cols, lr, weight_decay, scale, &kw, &ko);
  return launch_apply_bf16(static_cast<__nv_bfloat16 *>(param), static_cast<const __nv_bfloat16 *>(update), numel,
                           kw, ko, reinterpret_cast<cudaStream_t>(stream));
}

int muon_apply_update_f32(float *param, const float *update, int64_t batch, int64_t rows, int64_t cols, float lr,
                          float weight_decay, float scale, muon_stream_t stream) {
  if (batch < 0 || rows < 0 || cols < 0) return MUON_ERR_INVALID_ARG;
  const int64_t numel = batch * rows * cols;
  if (numel == 0) return MUON_OK;
  if (!param || !update || !isfinite(lr) || !isfinite(weight_decay) || !isfinite(scale)) return MUON_ERR_INVALID_ARG;
  float kw, ko;
  update_constants(rows, cols, lr, weight_decay, scale, &kw, &ko);
  return launch_apply_f32(param, update, numel, kw, ko, reinterpret_cast<cudaStream_t>(stream));
}

size_t muon_step_workspace_bytes(int64_t batch, int64_t rows, int64_t cols) {
  return muon_ns_workspace_bytes(batch, rows, cols);
}

// Orders the launch that writes W after `w_free` (if any) on stream s.
static int wait_param_free(cudaEvent_t w_free, cudaStream_t s) {
  if (w_free && cudaStreamWaitEvent(s, w_free, 0) != cudaSuccess) {
    cudaGetLastError();
    return MUON_ERR_CUDA;
  }
  return MUON_OK;
}

// momentum+norm -> iterations 1..steps-1 -> last iteration with the update.
// u lives in the second X buffer, which the rotation first writes in
// iteration 2, after iteration 1 has read u for the last time.  Only the last
// launch writes W; it waits for w_free first.
static int step_fused(__nv_bfloat16 *W, const __nv_bfloat16 *G, float *mom, const Workspace &w, int64_t batch,
                      int64_t rows, int64_t cols, float mu, int nesterov, int steps, const float *cf0,
                      int cf_stride, float eps, float kw, float ko, cudaEvent_t w_free, cudaStream_t s) {
  const int64_t mm = std::min(rows, cols), nn = std::max(rows, cols), per = rows * cols;
  const bool transposed = rows > cols;
  std::vector<IterPlan> plan;
  MUON_TRY(plan_ns(mm, steps, cf0, cf_stride, &plan));
  auto *x2 = static_cast<__nv_bfloat16 *>(w.x2);
  auto *lo = static_cast<uint8_t *>(w.lo);
  MUON_TRY(launch_momentum_norm_bf16(G, mom, x2, batch, per, mu, nesterov, eps, w.partial, w.inv, w.inv2, s));
  if (steps == 0) {
    MUON_TRY(launch_scale_bf16(x2, x2, batch, per, w.inv, s));
    MUON_TRY(wait_param_free(w_free, s));
    return launch_apply_bf16(W, x2, batch * per, kw, ko, s);
  }
  void *src = x2;
  for (int it = 0; it < steps; ++it) {
    const IterPlan &q = plan[it];
    MUON_TRY(ns_syrk(src, q.tin, w.a, q.store, batch, mm, nn, it == 0 ? w.inv2 : nullptr, q.syrk_mul, transposed, s));
    MUON_TRY(ns_poly(w.a, q.store, w.b, q.tin, batch, mm, q.poly_b, q.poly_c, s));
    const uint8_t *src_lo = reads_low_half(it, steps) ? lo : nullptr;
    const float *s1 = it == 0 ? w.inv : nullptr;
    if (it == steps - 1) {   // the last iteration's input carries no low half
      MUON_TRY(wait_param_free(w_free, s));
      return ns_axpy_apply(w.b, src, q.tin, W, batch, mm, nn, q.axpy_a, s1, q.axpy_mul, kw, ko, transposed, s);
    }
    void *dst = src == w.x1 ? w.x2 : w.x1;
    MUON_TRY(ns_axpy(w.b, src, q.tin, src_lo, q.lo_in, dst, q.store, writes_low_half(it, steps) ? lo : nullptr,
                     q.lo_out, batch, mm, nn, q.axpy_a, s1, q.axpy_mul, transposed, s));
    src = dst;
  }
  return MUON_OK;
}

// Checked arguments of both fused-step calls; cf holds (a, b, c) for step it
// at cf + it * cf_stride.
static int step_fused_entry(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows, int64_t cols,
                            float mu, int nesterov, int steps, const float *cf, int cf_stride, float eps, float lr,
                            float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                            cudaEvent_t w_free, cudaStream_t s) {
  if (!isfinite(mu) || !isfinite(lr) || !isfinite(weight_decay) || !isfinite(scale)) return MUON_ERR_INVALID_ARG;
  if (batch == 0) return MUON_OK;
  if (!grad || !momentum) return MUON_ERR_INVALID_ARG;
  if (rows % 8 || cols % 8 || !aligned16(param) || !aligned16(grad) || !aligned16(momentum))
    return MUON_ERR_UNSUPPORTED;
  std::vector<IterPlan> plan;
  MUON_TRY(plan_ns(std::min(rows, cols), steps, cf, cf_stride, &plan));
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MUON_ERR_INVALID_ARG;
  const int64_t mm = std::min(rows, cols), nn = std::max(rows, cols);
  const size_t need = ws_bytes(batch, mm, nn, 2);
  if (workspace && workspace_bytes < need) return MUON_ERR_NO_MEMORY;
  if (!device_error_word()) return MUON_ERR_CUDA;
  float kw, ko;
  update_constants(rows, cols, lr, weight_decay, scale, &kw, &ko);
  void *ws = workspace;
  if (!ws && (alloc_async(&ws, need, s) != cudaSuccess || !ws)) {
    cudaGetLastError();
    return MUON_ERR_NO_MEMORY;
  }
  int st = step_fused(static_cast<__nv_bfloat16 *>(param), static_cast<const __nv_bfloat16 *>(grad), momentum,
                      carve(ws, batch, mm, nn, 2), batch, rows, cols, mu, nesterov ? 1 : 0, steps, cf, cf_stride, eps,
                      kw, ko, w_free, s);
  if (!workspace && cudaFreeAsync(ws, s) != cudaSuccess && st == MUON_OK) st = MUON_ERR_CUDA;
  return st;
}

int muon_step_batched(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows, int64_t cols,
                      float mu, int nesterov, int steps, const float coeffs[3], float eps, float lr,
                      float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                      muon_stream_t stream) {
  MUON_TRY(check_ns_args(param, batch, rows, cols, steps, coeffs, eps));
  const float cf[3] = {coeffs[0], coeffs[1], coeffs[2]};
  return step_fused_entry(param, grad, momentum, batch, rows, cols, mu, nesterov, steps, cf, 0, eps, lr, weight_decay,
                          scale, workspace, workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int muon_step_batched_after(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows,
                            int64_t cols, float mu, int nesterov, int steps, const float coeffs[3], float eps,
                            float lr, float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                            muon_event_t param_free, muon_stream_t stream) {
  MUON_TRY(check_ns_args(param, batch, rows, cols, steps, coeffs, eps));
  const float cf[3] = {coeffs[0], coeffs[1], coeffs[2]};
  return step_fused_entry(param, grad, momentum, batch, rows, cols, mu, nesterov, steps, cf, 0, eps, lr, weight_decay,
                          scale, workspace, workspace_bytes, reinterpret_cast<cudaEvent_t>(param_free),
                          reinterpret_cast<cudaStream_t>(stream));
}

int muon_step_batched_schedule(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows,
                               int64_t cols, float mu, int nesterov, int steps, const float *coeffs, float eps,
                               float lr, float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                               muon_stream_t stream) {
  MUON_TRY(check_ns_args(param, batch, rows, cols, steps, coeffs, eps, 3 * (int64_t)steps));
  std::vector<float> cf(coeffs, coeffs + 3 * (size_t)steps);
  return step_fused_entry(param, grad, momentum, batch, rows, cols, mu, nesterov, steps, cf.data(), 3, eps, lr,
                          weight_decay, scale, workspace, workspace_bytes, nullptr,
                          reinterpret_cast<cudaStream_t>(stream));
}

static int adamw_consts(float lr, float beta1, float beta2, float eps, float wd, int64_t step, AdamWConsts *k) {
  if (step < 1 || !isfinite(lr) || !isfinite(eps) || !isfinite(wd) || !(beta1 >= 0.f && beta1 < 1.f) ||
      !(beta2 >= 0.f && beta2 < 1.f) || !(eps >= 0.f))
    return MUON_ERR_INVALID_ARG;
  const double t = (double)step;
  k->b1 = beta1;
  k->c1 = (float)(1.0 - (double)beta1);
  k->b2 = beta2;
  k->c2 = (float)(1.0 - (double)beta2);
  k->bc2 = (float)(1.0 - pow((double)beta2, t));
  k->step_size = (float)((double)lr / (1.0 - pow((double)beta1, t)));
  k->kw = (float)(1.0 - (double)lr * (double)wd);
  k->eps = eps;
  if (!(k->bc2 > 0.f) || !isfinite(k->step_size)) return MUON_ERR_INVALID_ARG;
  return MUON_OK;
}

int muon_adamw_update(void *param, const void *grad, float *exp_avg, float *exp_avg_sq, int64_t numel, float lr,
                      float beta1, float beta2, float eps, float weight_decay, int64_t step, muon_stream_t stream) {
  if (numel < 0) return MUON_ERR_INVALID_ARG;
  AdamWConsts k;
  MUON_TRY(adamw_consts(lr, beta1, beta2, eps, weight_decay, step, &k));
  if (numel == 0) return MUON_OK;
  if (!param || !grad || !exp_avg || !exp_avg_sq) return MUON_ERR_INVALID_ARG;
  return launch_adamw_bf16(static_cast<__nv_bfloat16 *>(param), static_cast<const __nv_bfloat16 *>(grad), exp_avg,
                           exp_avg_sq, numel, k, reinterpret_cast<cudaStream_t>(stream));
}

int muon_adamw_update_f32(float *param, const float *grad, float *exp_avg, float *exp_avg_sq, int64_t numel, float lr,
                          float beta1, float beta2, float eps, float weight_decay, int64_t step,
                          muon_stream_t stream) {
  if (numel < 0) return MUON_ERR_INVALID_ARG;
  AdamWConsts k;
  MUON_TRY(adamw_consts(lr, beta1, beta2, eps, weight_decay, step, &k));
  if (numel == 0) return MUON_OK;
  if (!param || !grad || !exp_avg || !exp_avg_sq) return MUON_ERR_INVALID_ARG;
  return launch_adamw_f32(param, grad, exp_avg, exp_avg_sq, numel, k, reinterpret_cast<cudaStream_t>(stream));
}

int muon_get_device_status(muon_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
  unsigned *p = device_error_word();
  if (!p) return MUON_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
  if (v && cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MUON_ERR_CUDA;
  if (v & kErrTimeout) return MUON_ERR_TIMEOUT;
  if (v & kErrDevice) return MUON_ERR_DEVICE;
  return MUON_OK;
}

const char *muon_status_string(int status) {
  switch (status) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_NO_MEMORY: return "MUON_ERR_NO_MEMORY";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
    case MUON_ERR_DEVICE: return "MUON_ERR_DEVICE";
    default: return "MUON_ERR_UNKNOWN";
  }
}

uint64_t muon_set_wait_timeout_ns(uint64_t timeout_ns) {
  return g_timeout_ns.exchange(timeout_ns ? timeout_ns : kDefaultTimeoutNs);
}

int muon_selftest_wait_timeout(uint64_t timeout_ns, muon_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MUON_ERR_INVALID_ARG;
  if (!device_error_word()) return MUON_ERR_CUDA;
  return selftest_wait(timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

int64_t muon_launch_count(void) { return g_launches.load(); }

int muon_inject_alloc_failures(int count) {
  if (count < 0) return MUON_ERR_INVALID_ARG;
  return g_fail_allocs.exchange(count);
}

int muon_trace_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_trace.on = true;
  return MUON_OK;
}

int muon_trace_end(muon_trace_entry *entries, int max_entries) {
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_trace.on = false;
    recs.swap(g_trace.recs);
    if (g_trace.pending_start) {
      g_trace.pool.push_back(g_trace.pending_start);
      g_trace.pending_start = nullptr;
    }
  }
  int64_t launches[kTraceKinds] = {};
  double ms[kTraceKinds] = {};
  int st = MUON_OK;
  for (const TraceRec &r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      st = MUON_ERR_CUDA;
    launches[r.kind] += 1;
    ms[r.kind] += t;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const TraceRec &r : recs) {
      g_trace.pool.push_back(r.start);
      g_trace.pool.push_back(r.stop);
    }
  }
  if (st != MUON_OK) return st;
  int kinds = 0;
  for (int k = 0; k < kTraceKinds; ++k) {
    if (!launches[k]) continue;
    if (entries && kinds < max_entries) entries[kinds] = {kTraceNames[k], launches[k], ms[k]};
    ++kinds;
  }
  return kinds;
}

}  // extern "C"
