// HBM-bound kernels of the Muon step: momentum, parameter update, per-matrix
// Frobenius norm, transpose and per-matrix scaling; and the AdamW update of
// the parameters Muon does not take.
//
// Source of the operations: "Training a 1T-Parameter MoE on EU public
// infrastructure with PyTorch and TorchTitan", section "FlexShard: Muon without
// communication" (one fp32 state per parameter; Newton-Schulz on whole
// matrices).  The momentum form, the normalisation and the update are the
// readings documented in muon.h.
//
// Access pattern: 16-byte vectors per thread (8 bf16 or 4 fp32), grid-stride
// loops over a grid sized in multiples of the SM count, and explicit
// round-to-nearest intrinsics so that nvcc cannot contract a multiply and an
// add into one fused operation (the results are specified per operation).
#include <algorithm>

#include "common.cuh"

namespace muon {
namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t items, int per_sm_blocks = 8) {
  int64_t want = (items + kThreads - 1) / kThreads;
  int64_t cap = (int64_t)num_sms() * per_sm_blocks;
  return (int)std::max<int64_t>(1, std::min(want, cap));
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__device__ __forceinline__ float mom_buf(float mu, float b, float g) { return __fadd_rn(__fmul_rn(mu, b), g); }
__device__ __forceinline__ float mom_u(float mu, float nb, float g, int nesterov) {
  return nesterov ? __fadd_rn(g, __fmul_rn(mu, nb)) : nb;
}

union Bf16x8 {
  uint4 v;
  __nv_bfloat162 h[4];
};

// ---------------------------------------------------------------- momentum
__global__ void momentum_bf16_vec(const uint4 *__restrict__ g8, float4 *__restrict__ buf4, uint4 *__restrict__ u8,
                                  int64_t nvec, float mu, int nesterov) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    Bf16x8 g;
    g.v = __ldcs(g8 + i);
    float4 b0 = __ldcs(buf4 + 2 * i), b1 = __ldcs(buf4 + 2 * i + 1);
    float gf[8], bf[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w}, uf[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 t = __bfloat1622float2(g.h[k]);
      gf[2 * k] = t.x;
      gf[2 * k + 1] = t.y;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      bf[k] = mom_buf(mu, bf[k], gf[k]);
      uf[k] = mom_u(mu, bf[k], gf[k], nesterov);
    }
    __stcs(buf4 + 2 * i, make_float4(bf[0], bf[1], bf[2], bf[3]));
    __stcs(buf4 + 2 * i + 1, make_float4(bf[4], bf[5], bf[6], bf[7]));
    Bf16x8 u;
#pragma unroll
    for (int k = 0; k < 4; ++k) u.h[k] = __floats2bfloat162_rn(uf[2 * k], uf[2 * k + 1]);
    __stcs(u8 + i, u.v);
  }
}

__global__ void momentum_bf16_scalar(const __nv_bfloat16 *__restrict__ g, float *__restrict__ buf,
                                     __nv_bfloat16 *__restrict__ u, int64_t begin, int64_t numel, float mu,
                                     int nesterov) {
  for (int64_t i = begin + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x) {
    float gf = __bfloat162float(g[i]);
    float nb = mom_buf(mu, buf[i], gf);
    buf[i] = nb;
    u[i] = __float2bfloat16_rn(mom_u(mu, nb, gf, nesterov));
  }
}

__global__ void momentum_f32_vec(const float4 *__restrict__ g4, float4 *__restrict__ buf4, float4 *__restrict__ u4,
                                 int64_t nvec, float mu, int nesterov) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    float4 g = __ldcs(g4 + i), b = __ldcs(buf4 + i);
    b.x = mom_buf(mu, b.x, g.x);
    b.y = mom_buf(mu, b.y, g.y);
    b.z = mom_buf(mu, b.z, g.z);
    b.w = mom_buf(mu, b.w, g.w);
    float4 u = make_float4(mom_u(mu, b.x, g.x, nesterov), mom_u(mu, b.y, g.y, nesterov),
                           mom_u(mu, b.z, g.z, nesterov), mom_u(mu, b.w, g.w, nesterov));
    __stcs(buf4 + i, b);
    __stcs(u4 + i, u);
  }
}

__global__ void momentum_f32_scalar(const float *__restrict__ g, float *__restrict__ buf, float *__restrict__ u,
                                    int64_t begin, int64_t numel, float mu, int nesterov) {
  for (int64_t i = begin + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x) {
    float nb = mom_buf(mu, buf[i], g[i]);
    buf[i] = nb;
    u[i] = mom_u(mu, nb, g[i], nesterov);
  }
}

// ---------------------------------------------------------------- update
__device__ __forceinline__ float upd(float kw, float ko, float w, float o) {
  return __fadd_rn(__fmul_rn(kw, w), __fmul_rn(ko, o));
}

__global__ void apply_bf16_vec(uint4 *__restrict__ w8, const uint4 *__restrict__ o8, int64_t nvec, float kw,
                               float ko) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    Bf16x8 w, o, r;
    w.v = __ldcs(w8 + i);
    o.v = __ldcs(o8 + i);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 wf = __bfloat1622float2(w.h[k]), of = __bfloat1622float2(o.h[k]);
      r.h[k] = __floats2bfloat162_rn(upd(kw, ko, wf.x, of.x), upd(kw, ko, wf.y, of.y));
    }
    __stcs(w8 + i, r.v);
  }
}

__global__ void apply_bf16_scalar(__nv_bfloat16 *__restrict__ w, const __nv_bfloat16 *__restrict__ o, int64_t begin,
                                  int64_t numel, float kw, float ko) {
  for (int64_t i = begin + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x)
    w[i] = __float2bfloat16_rn(upd(kw, ko, __bfloat162float(w[i]), __bfloat162float(o[i])));
}

__global__ void apply_f32_kernel(float *__restrict__ w, const float *__restrict__ o, int64_t numel, float kw,
                                 float ko) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x)
    w[i] = upd(kw, ko, w[i], o[i]);
}

// ---------------------------------------------------------------- AdamW
// Routers and embeddings take AdamW (two fp32 states per parameter); every
// fp32 operation is rounded separately in the order stated in muon.h.
__device__ __forceinline__ void adamw_elem(const AdamWConsts &k, float &w, float g, float &m, float &v) {
  m = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.c1, g));
  v = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.c2, __fmul_rn(g, g)));
  const float d = __fadd_rn(__fsqrt_rn(__fdiv_rn(v, k.bc2)), k.eps);
  w = __fsub_rn(__fmul_rn(k.kw, w), __fmul_rn(k.step_size, __fdiv_rn(m, d)));
}

__global__ void adamw_bf16_vec(uint4 *__restrict__ w8, const uint4 *__restrict__ g8, float4 *__restrict__ m4,
                               float4 *__restrict__ v4, int64_t nvec, AdamWConsts k) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    Bf16x8 w, g, r;
    w.v = __ldcs(w8 + i);
    g.v = __ldcs(g8 + i);
    float4 m0 = __ldcs(m4 + 2 * i), m1 = __ldcs(m4 + 2 * i + 1), v0 = __ldcs(v4 + 2 * i), v1 = __ldcs(v4 + 2 * i + 1);
    float mf[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float vf[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 wf = __bfloat1622float2(w.h[e]), gf = __bfloat1622float2(g.h[e]);
      adamw_elem(k, wf.x, gf.x, mf[2 * e], vf[2 * e]);
      adamw_elem(k, wf.y, gf.y, mf[2 * e + 1], vf[2 * e + 1]);
      r.h[e] = __floats2bfloat162_rn(wf.x, wf.y);
    }
    __stcs(w8 + i, r.v);
    __stcs(m4 + 2 * i, make_float4(mf[0], mf[1], mf[2], mf[3]));
    __stcs(m4 + 2 * i + 1, make_float4(mf[4], mf[5], mf[6], mf[7]));
    __stcs(v4 + 2 * i, make_float4(vf[0], vf[1], vf[2], vf[3]));
    __stcs(v4 + 2 * i + 1, make_float4(vf[4], vf[5], vf[6], vf[7]));
  }
}

__global__ void adamw_bf16_scalar(__nv_bfloat16 *__restrict__ w, const __nv_bfloat16 *__restrict__ g,
                                  float *__restrict__ m, float *__restrict__ v, int64_t begin, int64_t numel,
                                  AdamWConsts k) {
  for (int64_t i = begin + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x) {
    float wf = __bfloat162float(w[i]), mf = m[i], vf = v[i];
    adamw_elem(k, wf, __bfloat162float(g[i]), mf, vf);
    w[i] = __float2bfloat16_rn(wf);
    m[i] = mf;
    v[i] = vf;
  }
}

__global__ void adamw_f32_kernel(float *__restrict__ w, const float *__restrict__ g, float *__restrict__ m,
                                 float *__restrict__ v, int64_t numel, AdamWConsts k) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < numel; i += (int64_t)gridDim.x * blockDim.x) {
    float wf = w[i], mf = m[i], vf = v[i];
    adamw_elem(k, wf, g[i], mf, vf);
    w[i] = wf;
    m[i] = mf;
    v[i] = vf;
  }
}

// ---------------------------------------------------------------- norm
constexpr int kNormPartials = 64;

__device__ __forceinline__ float block_sum(float v) {
  __shared__ float red[kThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  }
  return t;  // valid in thread 0
}

// Each block sums the squares of one contiguous chunk of one matrix.
template <bool kVec>
__global__ void sumsq_bf16(const __nv_bfloat16 *__restrict__ x, int64_t per, float *__restrict__ partial) {
  const int64_t b = blockIdx.y;
  const __nv_bfloat16 *xb = x + b * per;
  const int64_t chunk = (per + kNormPartials - 1) / kNormPartials;
  int64_t lo = blockIdx.x * chunk, hi = min(per, lo + chunk);
  float acc0 = 0.f, acc1 = 0.f;
  if (kVec) {
    // chunk boundaries rounded to 8 elements (per % 8 == 0 on this path)
    lo = (lo + 7) & ~int64_t(7);
    hi = blockIdx.x == kNormPartials - 1 ? per : min(per, ((int64_t)(blockIdx.x + 1) * chunk + 7) & ~int64_t(7));
    const uint4 *v = reinterpret_cast<const uint4 *>(xb);
    for (int64_t i = lo / 8 + threadIdx.x; i < hi / 8; i += kThreads) {
      Bf16x8 t;
      t.v = __ldg(v + i);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(t.h[k]);
        acc0 = fmaf(f.x, f.x, acc0);
        acc1 = fmaf(f.y, f.y, acc1);
      }
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
      float f = __bfloat162float(xb[i]);
      acc0 = fmaf(f, f, acc0);
    }
  }
  float s = block_sum(acc0 + acc1);
  if (threadIdx.x == 0) partial[b * kNormPartials + blockIdx.x] = s;
}

// Momentum on one chunk of one matrix, fused with the sum of squares of the
// bf16 update it writes.  Block (j, b) covers exactly the elements and visits
// them in exactly the order of sumsq_bf16<true>'s block (j, b), so the partial
// sums, and hence the norms, equal those of momentum followed by the norm.
__global__ void momentum_sumsq_bf16(const uint4 *__restrict__ g8, float4 *__restrict__ buf4, uint4 *__restrict__ u8,
                                    int64_t per, float mu, int nesterov, float *__restrict__ partial) {
  const int64_t b = blockIdx.y;
  const int64_t chunk = (per + kNormPartials - 1) / kNormPartials;
  const int64_t lo = ((int64_t)blockIdx.x * chunk + 7) & ~int64_t(7);
  const int64_t hi =
      blockIdx.x == kNormPartials - 1 ? per : min(per, ((int64_t)(blockIdx.x + 1) * chunk + 7) & ~int64_t(7));
  const int64_t base = b * (per / 8);
  float acc0 = 0.f, acc1 = 0.f;
  for (int64_t i = base + lo / 8 + threadIdx.x; i < base + hi / 8; i += kThreads) {
    Bf16x8 g;
    g.v = __ldcs(g8 + i);
    float4 b0 = __ldcs(buf4 + 2 * i), b1 = __ldcs(buf4 + 2 * i + 1);
    float bf[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    Bf16x8 u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 gf = __bfloat1622float2(g.h[k]);
      bf[2 * k] = mom_buf(mu, bf[2 * k], gf.x);
      bf[2 * k + 1] = mom_buf(mu, bf[2 * k + 1], gf.y);
      u.h[k] = __floats2bfloat162_rn(mom_u(mu, bf[2 * k], gf.x, nesterov), mom_u(mu, bf[2 * k + 1], gf.y, nesterov));
      const float2 f = __bfloat1622float2(u.h[k]);
      acc0 = fmaf(f.x, f.x, acc0);
      acc1 = fmaf(f.y, f.y, acc1);
    }
    __stcs(buf4 + 2 * i, make_float4(bf[0], bf[1], bf[2], bf[3]));
    __stcs(buf4 + 2 * i + 1, make_float4(bf[4], bf[5], bf[6], bf[7]));
    u8[i] = u.v;  // read next by the first Newton-Schulz iteration: normal caching
  }
  float t = block_sum(acc0 + acc1);
  if (threadIdx.x == 0) partial[b * kNormPartials + blockIdx.x] = t;
}

__global__ void sumsq_f32(const float *__restrict__ x, int64_t per, float *__restrict__ partial) {
  const int64_t b = blockIdx.y;
  const float *xb = x + b * per;
  const int64_t chunk = (per + kNormPartials - 1) / kNormPartials;
  const int64_t lo = blockIdx.x * chunk, hi = min(per, lo + chunk);
  float acc = 0.f;
  for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) acc = fmaf(xb[i], xb[i], acc);
  float s = block_sum(acc);
  if (threadIdx.x == 0) partial[b * kNormPartials + blockIdx.x] = s;
}

// One warp per matrix: fixed-order sum of the partials, then 1/(sqrt + eps).
// A sum of squares that is not finite (an Inf or NaN in the input, or
// entries beyond ~1.8e19 whose squares overflow fp32) would make the factor
// 0 or NaN and the update silently zero or NaN; it sets kErrDevice in the
// error word, which muon_get_device_status reports as MUON_ERR_DEVICE.
__global__ void inv_norm_final(const float *__restrict__ partial, int64_t batch, float eps, float *__restrict__ inv,
                               float *__restrict__ inv2, unsigned *__restrict__ err) {
  const int64_t b = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= batch) return;
  float s = 0.f;
  for (int p = lane; p < kNormPartials; p += 32) s += partial[b * kNormPartials + p];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    if (!isfinite(s) && err) atomicOr(err, kErrDevice);
    float r = 1.0f / (sqrtf(s) + eps);
    inv[b] = r;
    if (inv2) inv2[b] = r * r;
  }
}

// ---------------------------------------------------------------- transpose
template <typename T>
__global__ void transpose_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t rows, int64_t cols) {
  __shared__ T tile[32][33];
  const int64_t b = blockIdx.z;
  const T *s = src + b * rows * cols;
  T *d = dst + b * rows * cols;
  const int64_t c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    int64_t r = r0 + threadIdx.y + k, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[threadIdx.y + k][threadIdx.x] = s[r * cols + c];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    int64_t c = c0 + threadIdx.y + k, r = r0 + threadIdx.x;  // output row c, column r
    if (r < rows && c < cols) d[c * rows + r] = tile[threadIdx.x][threadIdx.y + k];
  }
}

// ---------------------------------------------------------------- scaling
__global__ void scale_bf16(const __nv_bfloat16 *__restrict__ src, __nv_bfloat16 *__restrict__ dst, int64_t per,
                           const float *__restrict__ scale) {
  const int64_t b = blockIdx.y;
  const float f = scale[b];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per; i += (int64_t)gridDim.x * blockDim.x)
    dst[b * per + i] = __float2bfloat16_rn(f * __bfloat162float(src[b * per + i]));
}

__global__ void scale_f32(const float *__restrict__ src, float *__restrict__ dst, int64_t per,
                          const float *__restrict__ scale) {
  const int64_t b = blockIdx.y;
  const float f = scale[b];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per; i += (int64_t)gridDim.x * blockDim.x)
    dst[b * per + i] = f * src[b * per + i];
}

constexpr int64_t kMaxGridY = 65535;

}  // namespace

int norm_partials() { return kNormPartials; }

int launch_momentum_bf16(const __nv_bfloat16 *g, float *buf, __nv_bfloat16 *u, int64_t numel, float mu, int nesterov,
                         cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  int64_t done = 0;
  if (aligned16(g) && aligned16(buf) && aligned16(u)) {
    int64_t nvec = numel / 8;
    if (nvec > 0) {
      trace_before(kTraceMomentum, s);
      momentum_bf16_vec<<<grid_for(nvec), kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(g),
                                                            reinterpret_cast<float4 *>(buf),
                                                            reinterpret_cast<uint4 *>(u), nvec, mu, nesterov);
      int st = trace_after(kTraceMomentum, s);
      if (st) return st;
    }
    done = nvec * 8;
  }
  if (done < numel) {
    trace_before(kTraceMomentum, s);
    momentum_bf16_scalar<<<grid_for(numel - done), kThreads, 0, s>>>(g, buf, u, done, numel, mu, nesterov);
    return trace_after(kTraceMomentum, s);
  }
  return MUON_OK;
}

int launch_momentum_f32(const float *g, float *buf, float *u, int64_t numel, float mu, int nesterov, cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  int64_t done = 0;
  if (aligned16(g) && aligned16(buf) && aligned16(u)) {
    int64_t nvec = numel / 4;
    if (nvec > 0) {
      trace_before(kTraceMomentumF32, s);
      momentum_f32_vec<<<grid_for(nvec), kThreads, 0, s>>>(reinterpret_cast<const float4 *>(g),
                                                           reinterpret_cast<float4 *>(buf),
                                                           reinterpret_cast<float4 *>(u), nvec, mu, nesterov);
      int st = trace_after(kTraceMomentumF32, s);
      if (st) return st;
    }
    done = nvec * 4;
  }
  if (done < numel) {
    trace_before(kTraceMomentumF32, s);
    momentum_f32_scalar<<<grid_for(numel - done), kThreads, 0, s>>>(g, buf, u, done, numel, mu, nesterov);
    return trace_after(kTraceMomentumF32, s);
  }
  return MUON_OK;
}

int launch_apply_bf16(__nv_bfloat16 *w, const __nv_bfloat16 *o, int64_t numel, float kw, float ko, cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  int64_t done = 0;
  if (aligned16(w) && aligned16(o)) {
    int64_t nvec = numel / 8;
    if (nvec > 0) {
      trace_before(kTraceApply, s);
      apply_bf16_vec<<<grid_for(nvec), kThreads, 0, s>>>(reinterpret_cast<uint4 *>(w),
                                                         reinterpret_cast<const uint4 *>(o), nvec, kw, ko);
      int st = trace_after(kTraceApply, s);
      if (st) return st;
    }
    done = nvec * 8;
  }
  if (done < numel) {
    trace_before(kTraceApply, s);
    apply_bf16_scalar<<<grid_for(numel - done), kThreads, 0, s>>>(w, o, done, numel, kw, ko);
    return trace_after(kTraceApply, s);
  }
  return MUON_OK;
}

int launch_adamw_bf16(__nv_bfloat16 *w, const __nv_bfloat16 *g, float *m, float *v, int64_t numel,
                      const AdamWConsts &k, cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  int64_t done = 0;
  if (aligned16(w) && aligned16(g) && aligned16(m) && aligned16(v)) {
    int64_t nvec = numel / 8;
    if (nvec > 0) {
      trace_before(kTraceAdamW, s);
      adamw_bf16_vec<<<grid_for(nvec), kThreads, 0, s>>>(reinterpret_cast<uint4 *>(w), reinterpret_cast<const uint4 *>(g),
                                                         reinterpret_cast<float4 *>(m), reinterpret_cast<float4 *>(v),
                                                         nvec, k);
      int st = trace_after(kTraceAdamW, s);
      if (st) return st;
    }
    done = nvec * 8;
  }
  if (done < numel) {
    trace_before(kTraceAdamW, s);
    adamw_bf16_scalar<<<grid_for(numel - done), kThreads, 0, s>>>(w, g, m, v, done, numel, k);
    return trace_after(kTraceAdamW, s);
  }
  return MUON_OK;
}

int launch_adamw_f32(float *w, const float *g, float *m, float *v, int64_t numel, const AdamWConsts &k,
                     cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  trace_before(kTraceAdamW, s);
  adamw_f32_kernel<<<grid_for(numel), kThreads, 0, s>>>(w, g, m, v, numel, k);
  return trace_after(kTraceAdamW, s);
}

int launch_apply_f32(float *w, const float *o, int64_t numel, float kw, float ko, cudaStream_t s) {
  if (numel == 0) return MUON_OK;
  trace_before(kTraceApplyF32, s);
  apply_f32_kernel<<<grid_for(numel), kThreads, 0, s>>>(w, o, numel, kw, ko);
  return trace_after(kTraceApplyF32, s);
}

static int launch_final(const float *partial, int64_t batch, float eps, float *inv, float *inv2, cudaStream_t s) {
  trace_before(kTraceNormFinal, s);
  const int warps = 4;
  inv_norm_final<<<(unsigned)((batch + warps - 1) / warps), warps * 32, 0, s>>>(partial, batch, eps, inv, inv2,
                                                                                 device_error_word());
  return trace_after(kTraceNormFinal, s);
}

int launch_inv_norm_bf16(const __nv_bfloat16 *x, int64_t batch, int64_t per, float eps, float *partial, float *inv,
                         float *inv2, cudaStream_t s) {
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    dim3 grid(kNormPartials, (unsigned)nb);
    trace_before(kTraceNormPartial, s);
    if (per % 8 == 0 && aligned16(x))
      sumsq_bf16<true><<<grid, kThreads, 0, s>>>(x + b0 * per, per, partial + b0 * kNormPartials);
    else
      sumsq_bf16<false><<<grid, kThreads, 0, s>>>(x + b0 * per, per, partial + b0 * kNormPartials);
    int st = trace_after(kTraceNormPartial, s);
    if (st) return st;
  }
  return launch_final(partial, batch, eps, inv, inv2, s);
}

int launch_momentum_norm_bf16(const __nv_bfloat16 *g, float *buf, __nv_bfloat16 *u, int64_t batch, int64_t per,
                              float mu, int nesterov, float eps, float *partial, float *inv, float *inv2,
                              cudaStream_t s) {
  if (per % 8 || !aligned16(g) || !aligned16(buf) || !aligned16(u)) return MUON_ERR_UNSUPPORTED;
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    dim3 grid(kNormPartials, (unsigned)nb);
    trace_before(kTraceMomentumNorm, s);
    momentum_sumsq_bf16<<<grid, kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(g + b0 * per),
                                                  reinterpret_cast<float4 *>(buf + b0 * per),
                                                  reinterpret_cast<uint4 *>(u + b0 * per), per, mu, nesterov,
                                                  partial + b0 * kNormPartials);
    int st = trace_after(kTraceMomentumNorm, s);
    if (st) return st;
  }
  return launch_final(partial, batch, eps, inv, inv2, s);
}

int launch_inv_norm_f32(const float *x, int64_t batch, int64_t per, float eps, float *partial, float *inv, float *inv2,
                        cudaStream_t s) {
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    dim3 grid(kNormPartials, (unsigned)nb);
    trace_before(kTraceNormPartial, s);
    sumsq_f32<<<grid, kThreads, 0, s>>>(x + b0 * per, per, partial + b0 * kNormPartials);
    int st = trace_after(kTraceNormPartial, s);
    if (st) return st;
  }
  return launch_final(partial, batch, eps, inv, inv2, s);
}

template <typename T>
static int launch_transpose(const T *src, T *dst, int64_t batch, int64_t rows, int64_t cols, cudaStream_t s) {
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32), (unsigned)nb);
    trace_before(kTraceTranspose, s);
    transpose_kernel<T><<<grid, dim3(32, 8), 0, s>>>(src + b0 * rows * cols, dst + b0 * rows * cols, rows, cols);
    int st = trace_after(kTraceTranspose, s);
    if (st) return st;
  }
  return MUON_OK;
}

int launch_transpose_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int64_t batch, int64_t rows, int64_t cols,
                          cudaStream_t s) {
  return launch_transpose(src, dst, batch, rows, cols, s);
}

int launch_transpose_f32(const float *src, float *dst, int64_t batch, int64_t rows, int64_t cols, cudaStream_t s) {
  return launch_transpose(src, dst, batch, rows, cols, s);
}

int launch_scale_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int64_t batch, int64_t per, const float *scale,
                      cudaStream_t s) {
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    int gx = (int)std::max<int64_t>(1, std::min<int64_t>((per + kThreads - 1) / kThreads, 4 * num_sms()));
    trace_before(kTraceScale, s);
    scale_bf16<<<dim3(gx, (unsigned)nb), kThreads, 0, s>>>(src + b0 * per, dst + b0 * per, per, scale + b0);
    int st = trace_after(kTraceScale, s);
    if (st) return st;
  }
  return MUON_OK;
}

int launch_scale_f32(const float *src, float *dst, int64_t batch, int64_t per, const float *scale, cudaStream_t s) {
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxGridY) {
    int64_t nb = std::min(kMaxGridY, batch - b0);
    int gx = (int)std::max<int64_t>(1, std::min<int64_t>((per + kThreads - 1) / kThreads, 4 * num_sms()));
    trace_before(kTraceScale, s);
    scale_f32<<<dim3(gx, (unsigned)nb), kThreads, 0, s>>>(src + b0 * per, dst + b0 * per, per, scale + b0);
    int st = trace_after(kTraceScale, s);
    if (st) return st;
  }
  return MUON_OK;
}

}  // namespace muon
