// simt_gemm.cuh -- true-IEEE fp32 path: shared-memory-tiled FFMA GEMMs on
// the CUDA cores with the MLP's fused epilogues.  No tensor core, so no TF32:
// "[RFC] Testing Methodology for FP32 Convergence Tests on Fused
// SwiGLU/dSwiGLU Kernels" (Liger-Kernel #1383), "Root Cause" traces the fp32
// failures to TF32 matmuls, and "Approaches I tried" to the software-FMA
// path's shared-memory appetite on SM120 (a 64x64x16 fp32 tile pair here needs
// 8.5 KB, far inside sm_103a's 227 KB).
//
//   C[m, n] = sum_k A(m, k) B(n, k),  A(m, k) = A[m * sam + k * sak],
//                                     B(n, k) = B[n * sbn + k * sbk]
// Arbitrary element strides cover every K-major / MN-major operand of the
// six GEMMs.  A 64 x 64 output tile per 256-thread block, 4 x 4 per thread.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace swiglu {

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16, SG_THREADS = 256;

// Debug builds: the error word and the windows (operands, outputs) every
// element access is checked against; empty in release builds.
struct SimtCheck {
#ifdef SWIGLU_DEBUG
  int* err;
  DbgWin win;
#endif
};

// p[0], or 0 when a debug check rejects the address
__device__ __forceinline__ float simt_ld(const float* p, const SimtCheck& chk) {
  return SWIGLU_CHECK_PTR(chk.win, p, 4, chk.err) ? *p : 0.0f;
}

struct SimtOperand {
  const float* p;
  int64_t s_row;  // stride of the output-row index (m for A, n for B)
  int64_t s_k;    // stride of the contraction index
};

// Plain store: out[m * ld + n] = acc.
struct SimtEpiStore {
  float* out;
  int64_t ld;
  float scale = 1.0f;   // out = scale * acc ...
  int accumulate = 0;   // ... or, if nonzero, out + scale * acc
  __device__ __forceinline__ void apply(int m, int n, float acc, float,
                                        const SimtCheck& chk) const {
    float* o = out + (int64_t)m * ld + n;
    if (SWIGLU_CHECK_PTR(chk.win, o, 4, chk.err)) *o = accumulate ? *o + scale * acc : scale * acc;
  }
};

// sigma(g) = 1 / (1 + e^-g) and SiLU(g) = g sigma(g) with CUDA's expf and
// IEEE division, through t = e^-|g| (never overflows): for g < 0,
// sigma = t / (1 + t), so SiLU stays nonzero where its fp32 value is.
__device__ __forceinline__ float simt_sigmoid(float g) {
  const float t = expf(-fabsf(g));
  return g >= 0.0f ? 1.0f / (1.0f + t) : t / (1.0f + t);
}
__device__ __forceinline__ float simt_silu(float g) {
  const float t = expf(-fabsf(g));
  return g >= 0.0f ? g / (1.0f + t) : g * t / (1.0f + t);
}

// Gate/up: acc = X Wg^T, acc2 = u for hidden unit n; g = gate_mul * acc.
// Stores G = g, U (if g != null) and A = SiLU(g) * u.
struct SimtEpiSwiGLU {
  float* g;
  float* u;
  int64_t ld_gu;
  float* a;
  int64_t ld_a;
  float gate_mul = 1.0f;
  __device__ __forceinline__ void apply(int m, int n, float acc, float uv,
                                        const SimtCheck& chk) const {
    const float gv = gate_mul * acc;
    if (g != nullptr) {
      float* og = g + (int64_t)m * ld_gu + n;
      float* ou = u + (int64_t)m * ld_gu + n;
      if (SWIGLU_CHECK_PTR(chk.win, og, 4, chk.err)) *og = gv;
      if (SWIGLU_CHECK_PTR(chk.win, ou, 4, chk.err)) *ou = uv;
    }
    float* oa = a + (int64_t)m * ld_a + n;
    if (SWIGLU_CHECK_PTR(chk.win, oa, 4, chk.err)) *oa = simt_silu(gv) * uv;
  }
};

// Backward: acc = dY Wd for hidden unit n, dA = down_mul * acc; reads the
// stored G (= gate_mul X Wg^T), U and overwrites them with
// dG = dA * U * SiLU'(G) * gate_mul, dU = dA * SiLU(G).
struct SimtEpiDSwiGLU {
  float* g;
  float* u;
  int64_t ld;
  float gate_mul = 1.0f, down_mul = 1.0f;
  __device__ __forceinline__ void apply(int m, int n, float acc, float,
                                        const SimtCheck& chk) const {
    const int64_t o = (int64_t)m * ld + n;
    if (!(SWIGLU_CHECK_PTR(chk.win, g + o, 4, chk.err) &&
          SWIGLU_CHECK_PTR(chk.win, u + o, 4, chk.err)))
      return;
    const float da = down_mul * acc;
    const float gv = g[o], uv = u[o];
    const float s = simt_sigmoid(gv);
    u[o] = da * (gv * s);
    g[o] = da * uv * (s * (1.0f + gv * (1.0f - s)) * gate_mul);
  }
};

// DUAL: a second B operand (B2) accumulated alongside B; the epilogue gets
// both sums (used by the gate/up GEMM: B = Wg rows, B2 = Wu rows).
template <bool DUAL, class Epi>
__global__ void __launch_bounds__(SG_THREADS)
    simt_gemm_kernel(SimtOperand A, SimtOperand B, SimtOperand B2, int M, int N, int K, Epi epi,
                     SimtCheck chk) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  __shared__ float B2s[DUAL ? SG_BK : 1][SG_BN + 4];

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {}, acc2[4][4] = {};

  for (int k0 = 0; k0 < K; k0 += SG_BK) {
#pragma unroll
    for (int i = 0; i < (SG_BM * SG_BK) / SG_THREADS; ++i) {
      const int idx = threadIdx.x + i * SG_THREADS;
      const int r = idx / SG_BK, kk = idx % SG_BK;
      const int m = m0 + r, n = n0 + r, k = k0 + kk;
      As[kk][r] = (m < M && k < K) ? simt_ld(A.p + (int64_t)m * A.s_row + (int64_t)k * A.s_k, chk)
                                   : 0.0f;
      Bs[kk][r] = (n < N && k < K) ? simt_ld(B.p + (int64_t)n * B.s_row + (int64_t)k * B.s_k, chk)
                                   : 0.0f;
      if (DUAL)
        B2s[kk][r] = (n < N && k < K)
                         ? simt_ld(B2.p + (int64_t)n * B2.s_row + (int64_t)k * B2.s_k, chk)
                         : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
        if (DUAL) b2[i] = B2s[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (DUAL) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) epi.apply(m, n, acc[i][j], acc2[i][j], chk);
    }
}

}  // namespace swiglu
