// Internal declarations shared by the libmuon translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "muon.h"

namespace muon {

// Bits of the device error word.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrDevice = 2u;

// Kernel kinds known to the tracer (index into kTraceNames).
enum TraceKind : int {
  kTraceMomentum = 0,
  kTraceMomentumF32,
  kTraceNormPartial,
  kTraceNormFinal,
  kTraceTranspose,
  kTraceScale,
  kTraceSyrk,      // A = s^2 X X^T   (tensor cores)
  kTracePoly,      // B = b A + c A A (tensor cores)
  kTraceAxpy,      // X' = s (a X + B X) (tensor cores)
  kTraceApply,
  kTraceApplyF32,
  kTraceGemmF32,
  kTraceCopy,
  kTraceSelftest,
  kTraceAdamW,
  kTraceMomentumNorm,  // momentum fused with the per-matrix sum of squares
  kTraceAxpyApply,     // last iteration's X' = s (a X + B X) fused with W' = kw W + ko X'
  kTraceKinds
};

// Called around every kernel launch (cheap when tracing is off).
void trace_before(int kind, cudaStream_t s);
int trace_after(int kind, cudaStream_t s);   // checks cudaGetLastError; returns a muon_status

// Device address of the error word of the current device (never null after success).
unsigned *device_error_word();
unsigned long long wait_timeout_ns();
int num_sms();

// The library's own device allocations (stream-ordered on s): fails without a
// CUDA call while injected failures are pending (muon_inject_alloc_failures).
cudaError_t alloc_async(void **ptr, size_t bytes, cudaStream_t s);

// The argument, shape and coefficient checks of muon_ns_batched, in its order,
// without any CUDA call: MUON_OK when the call can go ahead.
int ns_precheck(const void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs, float eps);

// ---- elementwise / reduction kernels (elementwise.cu) ----
int launch_momentum_bf16(const __nv_bfloat16 *g, float *buf, __nv_bfloat16 *u, int64_t numel, float mu,
                         int nesterov, cudaStream_t s);
int launch_momentum_f32(const float *g, float *buf, float *u, int64_t numel, float mu, int nesterov,
                        cudaStream_t s);
int launch_apply_bf16(__nv_bfloat16 *w, const __nv_bfloat16 *o, int64_t numel, float kw, float ko,
                      cudaStream_t s);
int launch_apply_f32(float *w, const float *o, int64_t numel, float kw, float ko, cudaStream_t s);
// AdamW constants, formed in double on the host and rounded once to fp32
struct AdamWConsts {
  float b1, c1, b2, c2, bc2, step_size, kw, eps;
};
int launch_adamw_bf16(__nv_bfloat16 *w, const __nv_bfloat16 *g, float *m, float *v, int64_t numel,
                      const AdamWConsts &k, cudaStream_t s);
int launch_adamw_f32(float *w, const float *g, float *m, float *v, int64_t numel, const AdamWConsts &k,
                     cudaStream_t s);
// Per-matrix inverse norm: inv[b] = 1/(||X_b||_F + eps), inv2[b] = inv[b]^2.
// `partial` holds batch*norm_partials() floats of scratch.
int norm_partials();
int launch_inv_norm_bf16(const __nv_bfloat16 *x, int64_t batch, int64_t per, float eps, float *partial,
                         float *inv, float *inv2, cudaStream_t s);
// Momentum (as launch_momentum_bf16) on [batch][per] matrices, fused with the
// per-matrix inverse norm of the bf16 update u (as launch_inv_norm_bf16, with
// the same partial sums).  Requires per % 8 == 0 and 16-byte aligned arrays.
int launch_momentum_norm_bf16(const __nv_bfloat16 *g, float *buf, __nv_bfloat16 *u, int64_t batch, int64_t per,
                              float mu, int nesterov, float eps, float *partial, float *inv, float *inv2,
                              cudaStream_t s);
int launch_inv_norm_f32(const float *x, int64_t batch, int64_t per, float eps, float *partial, float *inv,
                        float *inv2, cudaStream_t s);
// dst[b] = src[b]^T for [batch][rows][cols] -> [batch][cols][rows]
int launch_transpose_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int64_t batch, int64_t rows,
                          int64_t cols, cudaStream_t s);
int launch_transpose_f32(const float *src, float *dst, int64_t batch, int64_t rows, int64_t cols,
                         cudaStream_t s);
// dst[b] = scale[b] * src[b] (per matrix of `per` elements); src may equal dst
int launch_scale_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int64_t batch, int64_t per,
                      const float *scale, cudaStream_t s);
int launch_scale_f32(const float *src, float *dst, int64_t batch, int64_t per, const float *scale,
                     cudaStream_t s);

// ---- tensor-core GEMMs of one Newton-Schulz iteration (gemm_tc.cu) ----
// 16-bit storage formats: the caller's matrices are bf16; what the iteration
// produces is stored in bf16 or in fp16 scaled by powers of two (see plan_ns
// in api.cu).
enum Fmt16 : int { kBF16 = 0, kF16 = 1, kE5M2 = 2 /* X's 8-bit low half only */ };
// All matrices are batched, densely packed, row-major; X is m x n (m <= n),
// stored as m x n or, with `transposed`, as its transpose (n x m).
// A = tout(mul * s2[b] * X X^T)   (s2 == nullptr: 1), upper triangle computed,
// mirrored; X of format tin (fp16 X gives fp16 A)
int ns_syrk(const void *X, int tin, void *A, int tout, int64_t batch, int64_t m, int64_t n, const float *s2,
            float mul, bool transposed, cudaStream_t s);
// B = tout(b*A + c*A A)   (A of format tin, symmetric), upper triangle computed,
// mirrored (bf16 A gives bf16 B)
int ns_poly(const void *A, int tin, void *B, int tout, int64_t batch, int64_t m, float b, float c, cudaStream_t s);
// Xn = tout(mul * s1[b] * (a*X + B X))   (s1 == nullptr: 1), with X = X + X_lo
// (B and X of format tin; X_lo e5m2 bytes times lo_in_mul) and the result
// split into Xn and Xn_lo = e5m2((result - Xn) * lo_out_mul); X_lo and Xn_lo
// may be null (zero low half / not wanted) and may be the same buffer (all
// of X, X_lo, Xn, Xn_lo in the same storage orientation)
int ns_axpy(const void *B, const void *X, int tin, const uint8_t *X_lo, float lo_in_mul, void *Xn, int tout,
            uint8_t *Xn_lo, float lo_out_mul, int64_t batch, int64_t m, int64_t n, float a, const float *s1, float mul,
            bool transposed, cudaStream_t s);
// The last iteration with the parameter update fused in (its input carries no
// low half): O = bf16(mul * s1[b] * (a*X + B X)) is not stored; W = bf16(kw*W +
// ko*O) in place, with W (bf16) stored in the same orientation as X.
int ns_axpy_apply(const void *B, const void *X, int tin, __nv_bfloat16 *W, int64_t batch, int64_t m, int64_t n,
                  float a, const float *s1, float mul, float kw, float ko, bool transposed, cudaStream_t s);
int selftest_wait(unsigned long long timeout_ns, cudaStream_t s);

// ---- fp32 SIMT GEMMs for the verification mode (gemm_f32.cu) ----
// mode 0: C = s2 * P P^T (P m x k);  mode 1: C = b*P + c*P P (P m x m);
// mode 2: C = s1 * (a*Q + P Q) (P m x m, Q m x n)
int gemm_f32(int mode, const float *P, const float *Q, float *C, int64_t batch, int64_t m, int64_t n,
             float a, float b, float c, const float *scale, cudaStream_t s);

}  // namespace muon
