// decode.cu -- sparse decode path ([SD] §3): per (token, slot) GEMVs that
// read topk_ids on the device and address only the selected expert's weights,
// the GLU between them and the weighted sum over local slots.
//
// GEMV grid (ceil(N/32), k, T), 8 warps per block, 4 output columns per warp.
// The block reads e = topk_ids[t, slot] first and returns block-uniformly,
// before any barrier, when e is not local ([SD] §3, first safety point). The
// activation row is staged to shared memory as fp32 with an XOR swizzle on
// 16-byte slots so that the per-lane float4 reads are free of bank conflicts.
// Each lane streams 16-byte weight chunks (16 e4m3 codes, or 32 e2m1 nibbles
// = one MXFP4 group with its UE8M0 scale) of 4 rows at once: 512 contiguous
// bytes per warp and row, coalesced.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kColsPerWarp = 4;
constexpr int kWarps = 8;

__device__ __forceinline__ int swz(int f) { return f ^ ((f >> 3) & 7); }

template <int WFMT>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(
    const uint16_t* __restrict__ xin, int x_per_slot, const int32_t* __restrict__ ids, int k,
    int expert_start, int n_local, const uint8_t* __restrict__ W, const float* __restrict__ wscale,
    const uint8_t* __restrict__ wsf, const uint16_t* __restrict__ bias, int N, int K,
    uint16_t* __restrict__ y) {
  extern __shared__ float4 xs4[];
  const int t = blockIdx.z, j = blockIdx.y;
  const int lid = ids[t * k + j] - expert_start;
  if (lid < 0 || lid >= n_local) return;  // block-uniform, before any barrier
  const uint16_t* xr = xin + (size_t)(x_per_slot ? (t * k + j) : t) * K;
  for (int f = threadIdx.x; f < K / 4; f += blockDim.x) {
    const uint2 p = __ldg(reinterpret_cast<const uint2*>(xr) + f);
    xs4[swz(f)] = make_float4(bf16_lo(p.x), bf16_hi(p.x), bf16_lo(p.y), bf16_hi(p.y));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int n0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kColsPerWarp;
  if (n0 >= N) return;
  constexpr int EPC = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? 16 : 32;  // elements per 16-byte chunk
  const int nchunk = K / EPC;
  const size_t row_bytes = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? (size_t)K : (size_t)K / 2;
  float acc[kColsPerWarp];
#pragma unroll
  for (int q = 0; q < kColsPerWarp; ++q) acc[q] = 0.0f;
  // Two 16-byte chunks per row and lane in flight: 8 loads per lane per step.
  for (int c0 = lane; c0 < nchunk; c0 += 64) {
    uint4 wv[2][kColsPerWarp];
    float sc[2][kColsPerWarp];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c0 + 32 * u;
#pragma unroll
      for (int q = 0; q < kColsPerWarp; ++q) {
        const int n = min(n0 + q, N - 1);
        wv[u][q] = (c < nchunk) ? __ldg(reinterpret_cast<const uint4*>(W + ((size_t)lid * N + n) * row_bytes) + c)
                                : make_uint4(0, 0, 0, 0);
        if (WFMT == MOE_WFMT_MXFP4_G32)
          sc[u][q] = (c < nchunk) ? pow2_f32((int)wsf[((size_t)lid * N + n) * (K / 32) + c] - 127) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c0 + 32 * u;
      if (c >= nchunk) break;
      float part[kColsPerWarp];
#pragma unroll
      for (int q = 0; q < kColsPerWarp; ++q) part[q] = 0.0f;
#pragma unroll
      for (int i = 0; i < EPC / 4; ++i) {
        const float4 xv = xs4[swz(c * (EPC / 4) + i)];
#pragma unroll
        for (int q = 0; q < kColsPerWarp; ++q) {
          const uint32_t* pw = &wv[u][q].x;
          float w0, w1, w2, w3;
          if (WFMT == MOE_WFMT_FP8_PER_EXPERT) {
            const uint32_t word = pw[i];
            const float2 a = e4m3x2_to_f32x2(word & 0xFFFFu);
            const float2 b = e4m3x2_to_f32x2(word >> 16);
            w0 = a.x; w1 = a.y; w2 = b.x; w3 = b.y;
          } else {
            const uint32_t word = pw[i >> 1] >> ((i & 1) * 16);
            const float2 a = e2m1x2_to_f32x2(word & 0xFFu);
            const float2 b = e2m1x2_to_f32x2((word >> 8) & 0xFFu);
            w0 = a.x; w1 = a.y; w2 = b.x; w3 = b.y;
          }
          part[q] = fmaf(w0, xv.x, part[q]);
          part[q] = fmaf(w1, xv.y, part[q]);
          part[q] = fmaf(w2, xv.z, part[q]);
          part[q] = fmaf(w3, xv.w, part[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < kColsPerWarp; ++q)
        acc[q] = (WFMT == MOE_WFMT_MXFP4_G32) ? fmaf(part[q], sc[u][q], acc[q]) : acc[q] + part[q];
    }
  }
#pragma unroll
  for (int q = 0; q < kColsPerWarp; ++q)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(kFull, acc[q], o);
  if (lane < kColsPerWarp && n0 + lane < N) {
    float a = acc[0];
#pragma unroll
    for (int q = 1; q < kColsPerWarp; ++q)
      if (lane == q) a = acc[q];
    const int n = n0 + lane;
    const float s = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? wscale[lid] : 1.0f;
    const float yv = fmaf(a, s, bf16_to_f32(bias[(size_t)lid * N + n]));
    y[((size_t)t * k + j) * N + n] = (uint16_t)f32_to_bf16_bits(yv);
  }
}

// GLU between the GEMVs: g = min(g, L), u = clamp(u, -L, L) when L > 0;
// act = (g * sigmoid(alpha g)) * (u + beta); local slots only.
__global__ void glu_kernel(const uint16_t* __restrict__ y1, const int32_t* __restrict__ ids, int T,
                           int k, int expert_start, int n_local, int I, int interleaved, float alpha,
                           float beta, float limit, uint16_t* __restrict__ act) {
  const long total = (long)T * k * I;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long)gridDim.x * blockDim.x) {
    const long r = idx / I;
    const int i = (int)(idx % I);
    const int lid = ids[r] - expert_start;
    if (lid < 0 || lid >= n_local) continue;
    const uint16_t* yr = y1 + (size_t)r * 2 * I;
    float g = bf16_to_f32(interleaved ? yr[2 * i] : yr[i]);
    float u = bf16_to_f32(interleaved ? yr[2 * i + 1] : yr[I + i]);
    if (limit > 0.0f) {
      g = fminf(g, limit);
      u = fminf(fmaxf(u, -limit), limit);
    }
    const float s = spec_sigmoid(__fmul_rn(alpha, g));
    act[(size_t)r * I + i] = (uint16_t)f32_to_bf16_bits(__fmul_rn(__fmul_rn(g, s), __fadd_rn(u, beta)));
  }
}

// out[t, h] = bf16(sum over local slots j, in order, of w[t,j] * y2[t,j,h]);
// non-local slots are skipped, never multiplied by zero.
__global__ void weighted_sum_kernel(const uint16_t* __restrict__ y2, const int32_t* __restrict__ ids,
                                    const float* __restrict__ topk_w, int T, int k, int expert_start,
                                    int n_local, int H, uint16_t* __restrict__ out) {
  const long total = (long)T * H;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / H);
    const int h = (int)(idx % H);
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int lid = ids[t * k + j] - expert_start;
      if (lid < 0 || lid >= n_local) continue;
      acc = __fmaf_rn(topk_w[t * k + j], bf16_to_f32(y2[((size_t)t * k + j) * H + h]), acc);
    }
    out[idx] = (uint16_t)f32_to_bf16_bits(acc);
  }
}

template <int WFMT>
cudaError_t gemv(const uint16_t* x, int x_per_slot, const moe_decode_args& a, const uint8_t* W,
                 const float* wscale, const uint8_t* wsf, const uint16_t* bias, int N, int K,
                 uint16_t* y, cudaStream_t st) {
  const dim3 grid((N + kWarps * kColsPerWarp - 1) / (kWarps * kColsPerWarp), a.k, a.T);
  const size_t smem = (size_t)K * sizeof(float);
  gemv_kernel<WFMT><<<grid, kWarps * 32, smem, st>>>(x, x_per_slot, a.topk_ids, a.k, a.expert_start,
                                                     a.num_local_experts, W, wscale, wsf, bias, N, K, y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const moe_decode_args& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t ce;
  const bool fp8 = a.wfmt == MOE_WFMT_FP8_PER_EXPERT;
  ce = fp8 ? gemv<MOE_WFMT_FP8_PER_EXPERT>(a.x, 0, a, a.w_gu, a.w_gu_scale, nullptr, a.b_gu, 2 * a.I, a.H, a.y1, st)
           : gemv<MOE_WFMT_MXFP4_G32>(a.x, 0, a, a.w_gu, nullptr, a.w_gu_sf, a.b_gu, 2 * a.I, a.H, a.y1, st);
  if (ce != cudaSuccess) return ce;
  {
    const long total = (long)a.T * a.k * a.I;
    glu_kernel<<<(int)lmin((total + 255) / 256, 4096), 256, 0, st>>>(
        a.y1, a.topk_ids, a.T, a.k, a.expert_start, a.num_local_experts, a.I,
        a.glu_layout == MOE_GLU_INTERLEAVED, a.glu_alpha, a.glu_beta, a.glu_limit, a.act);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;
  }
  ce = fp8 ? gemv<MOE_WFMT_FP8_PER_EXPERT>(a.act, 1, a, a.w_d, a.w_d_scale, nullptr, a.b_d, a.H, a.I, a.y2, st)
           : gemv<MOE_WFMT_MXFP4_G32>(a.act, 1, a, a.w_d, nullptr, a.w_d_sf, a.b_d, a.H, a.I, a.y2, st);
  if (ce != cudaSuccess) return ce;
  const long total = (long)a.T * a.H;
  weighted_sum_kernel<<<(int)lmin((total + 255) / 256, 4096), 256, 0, st>>>(
      a.y2, a.topk_ids, a.topk_w, a.T, a.k, a.expert_start, a.num_local_experts, a.H, a.out);
  return cudaGetLastError();
}

}  // namespace moe
