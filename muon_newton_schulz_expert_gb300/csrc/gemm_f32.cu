// fp32 SIMT GEMMs of the Newton-Schulz iteration for the verification mode.
//
// Same three contractions as the tensor-core path ("Training a 1T-Parameter
// MoE on EU public infrastructure with PyTorch and TorchTitan", section
// "FlexShard: Muon without communication": Newton-Schulz on whole matrices),
// written in plain fp32 fused multiply-adds on the CUDA cores: no TF32, no
// bf16 rounding, any shape.  Correctness reference only; not a fast path.
//   mode 0: C = s2 * P P^T       P m x K (K = n), C m x m
//   mode 1: C = b*P + c * P P    P m x m
//   mode 2: C = s1 * (a*Q + P Q) P m x m, Q m x n, C m x n
#include "common.cuh"

namespace muon {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <int MODE>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float *__restrict__ P, const float *__restrict__ Q,
                                                       float *__restrict__ C, int m, int n, float a, float b, float c,
                                                       const float *__restrict__ scale) {
  __shared__ float Ls[TK][TM + 4];
  __shared__ float Rs[TK][TN + 4];
  const int64_t bz = blockIdx.z;
  const int K = MODE == 0 ? n : m;            // reduction length
  const int ncols = MODE == 2 ? n : m;        // output columns
  const float *Pm = P + bz * (int64_t)m * (MODE == 0 ? n : m);
  const float *Qm = MODE == 2 ? Q + bz * (int64_t)m * n : nullptr;
  float *Cm = C + bz * (int64_t)m * ncols;
  const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    // left tile: L[i][k] = P[i][k]
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      int ii = e / TK, kk = e % TK;
      int i = i0 + ii, k = k0 + kk;
      Ls[kk][ii] = (i < m && k < K) ? Pm[(int64_t)i * K + k] : 0.f;
    }
    // right tile: R[k][j] = P[j][k] (mode 0), P[k][j] (mode 1), Q[k][j] (mode 2)
    for (int e = threadIdx.x; e < TN * TK; e += 256) {
      float v = 0.f;
      if (MODE == 0) {
        int jj = e / TK, kk = e % TK;
        int j = j0 + jj, k = k0 + kk;
        if (j < m && k < K) v = Pm[(int64_t)j * K + k];
        Rs[kk][jj] = v;
      } else {
        int kk = e / TN, jj = e % TN;
        int j = j0 + jj, k = k0 + kk;
        if (j < ncols && k < K) v = MODE == 1 ? Pm[(int64_t)k * m + j] : Qm[(int64_t)k * n + j];
        Rs[kk][jj] = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float l[4], r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        l[u] = Ls[kk][ty * 4 + u];
        r[u] = Rs[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(l[u], r[v], acc[u][v]);
    }
    __syncthreads();
  }
  const float sc = scale ? scale[bz] : 1.0f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= m) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j >= ncols) continue;
      float out;
      if (MODE == 0) {
        out = sc * acc[u][v];
      } else if (MODE == 1) {
        out = fmaf(c, acc[u][v], b * Pm[(int64_t)i * m + j]);
      } else {
        out = sc * fmaf(a, Qm[(int64_t)i * n + j], acc[u][v]);
      }
      Cm[(int64_t)i * ncols + j] = out;
    }
  }
}

}  // namespace

int gemm_f32(int mode, const float *P, const float *Q, float *C, int64_t batch, int64_t m, int64_t n, float a, float b,
             float c, const float *scale, cudaStream_t s) {
  const int64_t ncols = mode == 2 ? n : m;
  for (int64_t b0 = 0; b0 < batch; b0 += 65535) {
    const int64_t nb = batch - b0 < 65535 ? batch - b0 : 65535;
    dim3 grid((unsigned)((ncols + TN - 1) / TN), (unsigned)((m + TM - 1) / TM), (unsigned)nb);
    const float *sc = scale ? scale + b0 : nullptr;
    trace_before(kTraceGemmF32, s);
    if (mode == 0)
      gemm_f32_kernel<0><<<grid, 256, 0, s>>>(P + b0 * m * n, nullptr, C + b0 * m * m, (int)m, (int)n, a, b, c, sc);
    else if (mode == 1)
      gemm_f32_kernel<1><<<grid, 256, 0, s>>>(P + b0 * m * m, nullptr, C + b0 * m * m, (int)m, (int)n, a, b, c, sc);
    else
      gemm_f32_kernel<2><<<grid, 256, 0, s>>>(P + b0 * m * m, Q + b0 * m * n, C + b0 * m * n, (int)m, (int)n, a, b, c,
                                              sc);
    int st = trace_after(kTraceGemmF32, s);
    if (st) return st;
  }
  return MUON_OK;
}

}  // namespace muon
