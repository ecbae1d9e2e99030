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
// gated_rmsnorm_bf16_kernel: bf16 with V = 32, 64, 128 or 256: lanes take 8 values (one
// 16-byte load of o and of z), V / 8 lanes a row, so a warp covers 32 / (V / 8) rows a load;
// the arithmetic runs on fp32 pairs (packed FMA), SiLU(x) = x / (1 + e^-x) with e^-x as
// 2^(-x log2 e) on the hardware base-2 exponential and the division as a hardware reciprocal
// (as the conv's SiLU): about half the instructions of the per-element form, which was close
// to issue-bound.
// gated_rmsnorm_any_kernel: any V, lanes striding over the row twice.
// All are HBM-bound: 3 V dtype bytes per row (o and z in, y out).
#include <algorithm>

#include "common.cuh"
#include "conv_tap.cuh"

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

template <int LPR>
__global__ void __launch_bounds__(256, 4) gated_rmsnorm_bf16_kernel(const __nv_bfloat16 *o,
                                                                 const __nv_bfloat16 *__restrict__ z,
                                                                 const __nv_bfloat16 *__restrict__ w, int64_t rows,
                                                                 float eps, __nv_bfloat16 *y) {
  constexpr int V = 8 * LPR, RPW = 32 / LPR;  // values a row; rows a warp covers per load
  constexpr float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  uint64_t wv[4];
  if (w) unpack8p(*reinterpret_cast<const uint4 *>(w + li * 8), wv);
  else
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[i] = f2_pack(1.f, 1.f);
  const uint64_t neg_log2e = f2_pack(-kLog2e, -kLog2e), one = f2_pack(1.f, 1.f);
  // kRows row groups per pass, all their loads issued before the first is used (three keep
  // the kernel within 64 registers, four blocks an SM)
  constexpr int kRows = 3;
  const int64_t step = n_warps * RPW;
  for (int64_t g0 = warp_id * RPW + sub; g0 - sub < rows; g0 += kRows * step) {
    uint4 op[kRows], zp[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t r = g0 + i * step;
      if (r < rows) {
        op[i] = *reinterpret_cast<const uint4 *>(o + r * V + li * 8);
        zp[i] = *reinterpret_cast<const uint4 *>(z + r * V + li * 8);
      } else {
        op[i] = zp[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t r = g0 + i * step;
      uint64_t ov[4], zv[4];
      unpack8p(op[i], ov);
      unpack8p(zp[i], zv);
      uint64_t s2 = f2_mul(ov[0], ov[0]);
#pragma unroll
      for (int k = 1; k < 4; ++k) s2 = f2_fma(ov[k], ov[k], s2);
      float sa, sb;
      f2_unpack(s2, sa, sb);
      float ss = sa + sb;
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv = 1.f / sqrtf(ss * (1.f / V) + eps);
      const uint64_t sc = f2_pack(inv, inv);
      uint64_t yv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float e0, e1, d0, d1;
        f2_unpack(f2_mul(zv[k], neg_log2e), e0, e1);
        f2_unpack(f2_add(f2_pack(hw_exp2(e0), hw_exp2(e1)), one), d0, d1);
        const uint64_t gate = f2_mul(zv[k], f2_pack(hw_rcp(d0), hw_rcp(d1)));  // silu(z)
        yv[k] = f2_mul(f2_mul(f2_mul(ov[k], sc), wv[k]), gate);
      }
      if (r < rows) *reinterpret_cast<uint4 *>(y + r * V + li * 8) = pack8p(yv);
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
  if constexpr (sizeof(T) == 2) {
    if (al && (!w || aligned(w, 16))) {
      const __nv_bfloat16 *ob = (const __nv_bfloat16 *)o, *zb = (const __nv_bfloat16 *)z,
                          *wb = (const __nv_bfloat16 *)w;
      __nv_bfloat16 *yb = (__nv_bfloat16 *)y;
      const int lpr = V / 8;
      const int64_t rows_per_block = 8 * (32 / std::max(lpr, 1));
      const unsigned g = (unsigned)std::min<int64_t>((rows + rows_per_block - 1) / rows_per_block, (int64_t)sms * 8);
      switch (V) {
        case 32: gated_rmsnorm_bf16_kernel<4><<<g, 256, 0, st>>>(ob, zb, wb, rows, eps, yb); return launch_status();
        case 64: gated_rmsnorm_bf16_kernel<8><<<g, 256, 0, st>>>(ob, zb, wb, rows, eps, yb); return launch_status();
        case 128: gated_rmsnorm_bf16_kernel<16><<<g, 256, 0, st>>>(ob, zb, wb, rows, eps, yb); return launch_status();
        case 256: gated_rmsnorm_bf16_kernel<32><<<g, 256, 0, st>>>(ob, zb, wb, rows, eps, yb); return launch_status();
        default: break;
      }
    }
  }
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
