// norm.cu -- gated RMS norm of the recurrent core's output, the layer's "+ norm" after
// chunk_gated_delta_rule ("[v1] support GDN Ulysses cp", Design; z is one of the layer's
// per-token components).  The pages give no formula; the reading taken is, per row r of
// V values (a token's v-head),
//     y[r, v] = o[r, v] / sqrt(mean_v o[r, :]^2 + eps) * w[v] * silu(z[r, v]).
//
// gated_rmsnorm_kernel: one warp per row (grid-stride over rows, four rows' loads in
// flight per warp); for V = 32 E with E in {1, 2, 4, 8}, lane l holds the E consecutive
// values l E .. l E + E - 1 of o and z, each one aligned vector load, and the sum of squares
// is a warp reduction.  Every lane writes only the values it read, so y may alias o.
// gated_rmsnorm_any_kernel: any V, lanes striding over the row twice.
// Both are HBM-bound: 3 V dtype bytes per row (o and z in, y out).
#include <algorithm>

#include "common.cuh"

using namespace gdn;

namespace {

template <typename T, int E>
struct alignas(E * sizeof(T) >= 16 ? 16 : E * sizeof(T)) Pack {
  T v[E];
};

__device__ __forceinline__ float silu_gate(float z) { return __fdividef(z, 1.f + __expf(-z)); }

template <typename T, int E>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const T *o, const T *__restrict__ z,
                                                            const T *__restrict__ w, int64_t rows, float eps,
                                                            T *y) {
  constexpr int V = 32 * E;
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float wv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) wv[e] = w ? to_f32<T>(w[lane * E + e]) : 1.f;
  // kRows rows per pass, all their loads issued before the first is used
  constexpr int kRows = 4;
  for (int64_t r0 = first; r0 < rows; r0 += kRows * stride) {
    Pack<T, E> op[kRows], zp[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t r = r0 + i * stride;
      if (r < rows) {
        op[i] = *reinterpret_cast<const Pack<T, E> *>(o + r * V + lane * E);
        zp[i] = *reinterpret_cast<const Pack<T, E> *>(z + r * V + lane * E);
      }
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t r = r0 + i * stride;
      if (r >= rows) break;
      float ov[E], ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        ov[e] = to_f32<T>(op[i].v[e]);
        ss = fmaf(ov[e], ov[e], ss);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv = 1.f / sqrtf(ss * (1.f / V) + eps);
      Pack<T, E> yp;
#pragma unroll
      for (int e = 0; e < E; ++e) yp.v[e] = from_f32<T>(ov[e] * inv * wv[e] * silu_gate(to_f32<T>(zp[i].v[e])));
      *reinterpret_cast<Pack<T, E> *>(y + r * V + lane * E) = yp;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) gated_rmsnorm_any_kernel(const T *o, const T *__restrict__ z,
                                                                const T *__restrict__ w, int64_t rows, int V,
                                                                float eps, T *y) {
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = first; r < rows; r += stride) {
    const T *orow = o + r * V;
    float ss = 0.f;
    for (int v = lane; v < V; v += 32) {
      const float x = to_f32<T>(orow[v]);
      ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.f / sqrtf(ss / (float)V + eps);
    for (int v = lane; v < V; v += 32) {
      const float wv = w ? to_f32<T>(w[v]) : 1.f;
      y[r * V + v] = from_f32<T>(to_f32<T>(orow[v]) * inv * wv * silu_gate(to_f32<T>(z[r * V + v])));
    }
  }
}

template <typename T>
gdn_status launch_norm(const void *o, const void *z, const void *w, int64_t rows, int V, float eps, void *y,
                       cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int64_t want = (rows + 7) / 8;  // 8 rows (warps) per block of 256
  const unsigned grid = (unsigned)std::min<int64_t>(want, (int64_t)sms * 8);
  const size_t vb = (size_t)V * sizeof(T);
  const bool al = aligned(o, 16) && aligned(z, 16) && aligned(y, 16);
  const T *op = (const T *)o, *zp = (const T *)z, *wp = (const T *)w;
  T *yp = (T *)y;
  if (al && vb % 16 == 0) {
    switch (V) {
      case 32: gated_rmsnorm_kernel<T, 1><<<grid, 256, 0, st>>>(op, zp, wp, rows, eps, yp); return launch_status();
      case 64: gated_rmsnorm_kernel<T, 2><<<grid, 256, 0, st>>>(op, zp, wp, rows, eps, yp); return launch_status();
      case 128: gated_rmsnorm_kernel<T, 4><<<grid, 256, 0, st>>>(op, zp, wp, rows, eps, yp); return launch_status();
      case 256: gated_rmsnorm_kernel<T, 8><<<grid, 256, 0, st>>>(op, zp, wp, rows, eps, yp); return launch_status();
      default: break;
    }
  }
  gated_rmsnorm_any_kernel<T><<<grid, 256, 0, st>>>(op, zp, wp, rows, V, eps, yp);
  return launch_status();
}

}  // namespace

extern "C" gdn_status gdn_gated_rmsnorm(const void *o, const void *z, const void *w, int32_t dtype, int64_t n_rows,
                                        int32_t V, float eps, void *y, void *stream) {
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (n_rows < 0 || V < 1 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (n_rows == 0) return GDN_OK;
  if (!o || !z || !y) return GDN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == GDN_BF16) return launch_norm<__nv_bfloat16>(o, z, w, n_rows, V, eps, y, st);
  return launch_norm<float>(o, z, w, n_rows, V, eps, y, st);
}
