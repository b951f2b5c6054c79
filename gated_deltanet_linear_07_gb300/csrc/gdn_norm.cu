// Gated RMSNorm of the layer output (the DeltaNet "gated norm"):
//   y_j = o_j / sqrt(mean_j o_j^2 + eps) * w_j * SiLU(z_j)
// over each row of d_v values (one token, one value head).  The weight is
// applied as stored (oxydllm 0.0.0-alpha.12.2 release notes, New Features,
// "GGUF qwen35 architecture": this norm alone carries no pre-added +1).
//
// HBM-bound: a row is read twice (o, z) and written once.  A row is handled
// by LPR = d_v / VEC consecutive lanes, VEC elements (16 bytes) each; the sum
// of squares is reduced over those lanes with shuffles.
#include "gdn_common.cuh"

namespace gdn {

template <typename IO>
struct NormVec;
template <>
struct NormVec<float> {
  static constexpr int VEC = 4;
  __device__ static void load(const void* p, float (&v)[4]) {
    const float4 f = __ldcs(reinterpret_cast<const float4*>(p));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
  __device__ static void store(void* p, const float (&v)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  }
};
template <>
struct NormVec<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ static void load(const void* p, float (&v)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(void* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
  }
};

template <typename IO, int LPR>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const float* __restrict__ weight,
                                                            float eps, const void* o, const void* z,
                                                            int64_t rows, void* y) {
  using V = NormVec<IO>;
  constexpr int VEC = V::VEC, DV = VEC * LPR;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = t / LPR;
  const int part = (int)(t % LPR);
  // every lane of a row group takes part in the shuffles; rows past the end
  // compute on zeros and store nothing
  const bool live = row < rows;
  const size_t off = (size_t)(live ? row : 0) * DV + (size_t)part * VEC;
  float ov[VEC], zv[VEC];
  V::load(reinterpret_cast<const IO*>(o) + off, ov);
  V::load(reinterpret_cast<const IO*>(z) + off, zv);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) ss = fmaf(ov[i], ov[i], ss);
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m, LPR);
  const float inv = rsqrtf(ss * (1.0f / DV) + eps);
  const float4* w4 = reinterpret_cast<const float4*>(weight + part * VEC);
  float yv[VEC];
#pragma unroll
  for (int i = 0; i < VEC; i += 4) {
    const float4 w = __ldg(w4 + i / 4);
    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // SiLU(z) = z / (1 + 2^(-z log2 e)) with the exponential and the
      // quotient on the special-function unit: relative accuracy of a few ulp
      // for every z (the form h + h tanh(h) loses it for negative z, where
      // the two terms cancel); -> 0 for z -> -inf, z for z -> +inf.
      const float zk = zv[i + k];
      float e;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * zk));
      yv[i + k] = ov[i + k] * inv * wv[k] * __fdividef(zk, 1.0f + e);
    }
  }
  if (live) V::store(reinterpret_cast<IO*>(y) + off, yv);
}

template <typename IO>
static cudaError_t launch_norm(const float* weight, float eps, const void* o, const void* z,
                               int64_t rows, int d_v, void* y, cudaStream_t s) {
  constexpr int VEC = NormVec<IO>::VEC;
  const int lpr = d_v / VEC;
  const int64_t threads = rows * lpr;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  switch (lpr) {
#define GDN_NORM_CASE(N)                                                              \
  case N:                                                                             \
    gated_rmsnorm_kernel<IO, N><<<grid, 256, 0, s>>>(weight, eps, o, z, rows, y);     \
    break;
    GDN_NORM_CASE(2)
    GDN_NORM_CASE(4)
    GDN_NORM_CASE(8)
    GDN_NORM_CASE(16)
    GDN_NORM_CASE(32)
#undef GDN_NORM_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_gated_rmsnorm(const float* weight, float eps, const void* o, const void* z,
                                     int64_t rows, int d_v, int io, void* y, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  return io == GDN_BF16 ? gdn::launch_norm<__nv_bfloat16>(weight, eps, o, z, rows, d_v, y, s)
                        : gdn::launch_norm<float>(weight, eps, o, z, rows, d_v, y, s);
}
