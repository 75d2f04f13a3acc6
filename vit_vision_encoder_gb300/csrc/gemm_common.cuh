// Pieces of the tcgen05 GEMM shared by the one-CTA kernel (gemm.cu) and the
// CTA-pair kernel (gemm_pair.cu): the kernel parameters, the tile order and
// the packed erf-GELU of the epilogue.  Included inside namespace
// dsvit::{anonymous} of each translation unit, after internal.h and ptx.cuh.
#pragma once

struct GemmParams {
  int M, N, K;
  bf16* out;          // read by the residual epilogue; written through tmC
  const bf16* bias;
  const int* rowpos;
  const float* rope_cs;
  int* status;
  int n_fast;         // tile order: 1 = n-block fastest, 0 = m-block fastest
};

// n-block-fastest order when the A operand would not stay in L2 between the
// passes over its n-blocks.
int tile_order(int64_t M, int K) { return M * K * 2 > (int64_t{40} << 20) ? 1 : 0; }

// GELU(x) = x Phi(x), Phi from erf ("End-to-end results and their limits":
// the erf form).  erf by Abramowitz & Stegun 7.1.26 (Hastings): for z >= 0,
// erfc(z) ~ q = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2) with
// t = 1 / (1 + p z), |erf error| <= 1.5e-7; then 2 Phi(x) = 2 - q for x >= 0
// and q for x < 0 (z = |x| / sqrt 2), so the negative tail keeps its relative
// precision.  Over [-10, 10] the GELU error is below 2.2e-7 absolute and
// 1.7e-4 relative wherever |GELU| > 1e-3.  Two elements per call, on packed
// f32x2 arithmetic; reciprocal and exp2 are the MUFU approximations.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void gelu_erf2(float& x0, float& x1) {
  const float kP = 0.3275911f;
  const uint64_t a5 = pk2(1.061405429f, 1.061405429f), a4 = pk2(-1.453152027f, -1.453152027f);
  const uint64_t a3 = pk2(1.421413741f, 1.421413741f), a2 = pk2(-0.284496736f, -0.284496736f);
  const uint64_t a1 = pk2(0.254829592f, 0.254829592f);
  const float z0 = fabsf(x0) * 0.70710678118654752f, z1 = fabsf(x1) * 0.70710678118654752f;
  const uint64_t z = pk2(z0, z1);
  float d0, d1;
  upk2(fma2(pk2(kP, kP), z, pk2(1.f, 1.f)), d0, d1);
  const uint64_t t = pk2(rcp_approx(d0), rcp_approx(d1));
  uint64_t poly = fma2(a5, t, a4);
  poly = fma2(poly, t, a3);
  poly = fma2(poly, t, a2);
  poly = fma2(poly, t, a1);
  poly = mul2(poly, t);
  float w0, w1;   // -z^2 log2(e)
  upk2(mul2(mul2(z, z), pk2(-1.4426950408889634f, -1.4426950408889634f)), w0, w1);
  float q0, q1;
  upk2(mul2(poly, pk2(ex2_approx(w0), ex2_approx(w1))), q0, q1);
  const float p0 = x0 >= 0.f ? 2.f - q0 : q0, p1 = x1 >= 0.f ? 2.f - q1 : q1;   // 2 Phi
  float g0, g1;
  upk2(mul2(mul2(pk2(x0, x1), pk2(0.5f, 0.5f)), pk2(p0, p1)), g0, g1);
  x0 = g0;
  x1 = g1;
}

// Tile order.  n-block fastest: the CTAs resident at one time cover few row
// blocks of A, each read from DRAM once and shared through L2 by all the
// n-blocks of its row (m-block-fastest order re-read the 75 MB A of the FC2
// shape from DRAM once per n-block column).  m-block fastest: the resident
// CTAs share few B tiles, which suits an A that stays in L2 anyway.
__device__ __forceinline__ int tile_mb(int tile, int num_m, int num_n, int n_fast) {
  return n_fast ? tile / num_n : tile % num_m;
}
__device__ __forceinline__ int tile_nb(int tile, int num_m, int num_n, int n_fast) {
  return n_fast ? tile % num_n : tile / num_m;
}
