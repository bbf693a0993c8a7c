// act_quant.cu -- live-row SiLU*mul + e4m3 quantisation with packed UE8M0
// group scales ([LR] §2-3, [DG] §2.4.1).
//
// Live launch: grid (1, gy, E) with the expert on axis z. Block (e, y) reads
// start[e] = align_up(end[e-1], A) and end[e] from the device-side endpoint
// tensor and walks the work items of [start[e], end[e)) with a grid-stride
// loop; rows outside the live ranges are never read or written. Dense
// fallback (no endpoints): grid (1, gy, 1) over every row of the buffer.
//
// Work item = (row, packed scale word w): the 512 columns of groups
// 4w..4w+3. One warp per item, 16 columns per lane (two uint4 loads from the
// gate half, two from the up half); a group of 128 columns is 8 lanes, its
// amax a 3-step xor reduction; lane 0 assembles the four scale bytes into the
// int32 word of the MN-major scale array. SiTU ([DG] §2.4.1) reads gate' and
// up' from two per-context tables over all bf16 patterns.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kThreads = 256;

// kAct: 0 SiLU, 1 SiLU with the clamp, 2 SiTU (situ_tbl: gate' then up'
// tables over all bf16 patterns, for the context's beta_s / beta_l).
template <bool kLive, int kAct>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint16_t* __restrict__ gateup,
                                                             uint8_t* __restrict__ out,
                                                             int32_t* __restrict__ out_sf,
                                                             const int32_t* __restrict__ ends, int E,
                                                             int A, int M_alloc, int I, int ld_sf,
                                                             float limit, const float* __restrict__ silu_tbl,
                                                             const float* __restrict__ situ_tbl,
                                                             bool g32, uint32_t* err) {
  constexpr bool kClamp = kAct == 1;
  const float silu_limit = kClamp ? spec_silu(limit) : 0.0f;
  int r0 = 0, r1 = M_alloc;
  if (kLive) {
    const int e = blockIdx.z;
    r1 = ends[e];
    r0 = (e == 0) ? 0 : (int)align_up64(ends[e - 1], A);
    if (r1 < r0 || r1 > M_alloc) {
      if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(err, MOE_DEVERR_ENDPOINTS);
      return;
    }
  }
  const int G = I / 128;
  const int G4 = (G + 3) / 4;
  const int lane = threadIdx.x & 31;
  const long n_items = (long)(r1 - r0) * G4;
  const long stride = (long)gridDim.x * gridDim.y * (kThreads / 32);
  for (long item = ((long)blockIdx.y * gridDim.x + blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
       item < n_items; item += stride) {
    const int row = r0 + (int)(item / G4);
    const int w = (int)(item % G4);
    const int col = w * 512 + lane * 16;
    const bool active = col < I;
    float h[16];
    float amax = 0.0f;
    uint4 g0 = make_uint4(0, 0, 0, 0), g1 = g0, u0 = g0, u1 = g0;
    if (active) {
      const uint16_t* g = gateup + (size_t)row * 2 * I + col;
      g0 = __ldg(reinterpret_cast<const uint4*>(g));
      g1 = __ldg(reinterpret_cast<const uint4*>(g + 8));
      u0 = __ldg(reinterpret_cast<const uint4*>(g + I));
      u1 = __ldg(reinterpret_cast<const uint4*>(g + I + 8));
    }
    const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    if (active) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ga = bf16_lo(gw[i]), gb = bf16_hi(gw[i]);
        float ua = bf16_lo(uw[i]), ub = bf16_hi(uw[i]);
        float sa, sb;
        if (kAct == 2) {
          sa = __ldg(situ_tbl + (gw[i] & 0xFFFFu));
          sb = __ldg(situ_tbl + (gw[i] >> 16));
          ua = __ldg(situ_tbl + 65536 + (uw[i] & 0xFFFFu));
          ub = __ldg(situ_tbl + 65536 + (uw[i] >> 16));
        } else {
          if (kClamp) {
            ua = fminf(fmaxf(ua, -limit), limit);
            ub = fminf(fmaxf(ub, -limit), limit);
          }
          sa = silu_of_bf16<kClamp>(silu_tbl, gw[i], ga, limit, silu_limit);
          sb = silu_of_bf16<kClamp>(silu_tbl, gw[i] >> 16, gb, limit, silu_limit);
        }
        const float2 hh = mul2(make_float2(sa, sb), make_float2(ua, ub));
        h[2 * i] = hh.x;
        h[2 * i + 1] = hh.y;
        amax = fmaxf(amax, fmaxf(fabsf(hh.x), fabsf(hh.y)));
      }
    }
#pragma unroll
    // 8 lanes per 128-column group, or 2 per 32-column group (MXFP8)
    for (int o = g32 ? 1 : 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const uint32_t b = active ? group_scale_byte(amax) : 0u;
    if (active) {
      const float sc = pow2_f32(127 - (int)b);
      uint4 q;
      uint32_t* qw = &q.x;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qw[i] = e4m3x2_satfinite(__fmul_rn(h[4 * i], sc), __fmul_rn(h[4 * i + 1], sc)) |
                (e4m3x2_satfinite(__fmul_rn(h[4 * i + 2], sc), __fmul_rn(h[4 * i + 3], sc)) << 16);
      *reinterpret_cast<uint4*>(out + (size_t)row * I + col) = q;
    }
    if (g32) {
      // one word per 128 columns (8 lanes): the bytes of lanes 8q, 8q+2, 8q+4, 8q+6
      const int q0 = lane & ~7;
      const uint32_t word = __shfl_sync(kFull, b, q0) | (__shfl_sync(kFull, b, q0 + 2) << 8) |
                            (__shfl_sync(kFull, b, q0 + 4) << 16) | (__shfl_sync(kFull, b, q0 + 6) << 24);
      if ((lane & 7) == 0 && active) out_sf[(size_t)(4 * w + (lane >> 3)) * ld_sf + row] = (int32_t)word;
    } else {
      const uint32_t b0 = __shfl_sync(kFull, b, 0), b1 = __shfl_sync(kFull, b, 8);
      const uint32_t b2 = __shfl_sync(kFull, b, 16), b3 = __shfl_sync(kFull, b, 24);
      if (lane == 0) out_sf[(size_t)w * ld_sf + row] = (int32_t)(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
    }
  }
}

template <bool kLive>
cudaError_t launch_kind(const uint16_t* gateup, uint8_t* out, int32_t* out_sf, const int32_t* ends,
                        int E, int A, int M_alloc, int I, int kind, float limit, const float* silu_tbl,
                        const float* situ_tbl, bool g32, dim3 grid, uint32_t* err, cudaStream_t st) {
  const int ld = (int)align_up64(M_alloc, 4);
  if (kind == MOE_ACT_SILU_CLAMP)
    act_quant_kernel<kLive, 1><<<grid, kThreads, 0, st>>>(gateup, out, out_sf, ends, E, A, M_alloc, I, ld, limit,
                                                        silu_tbl, situ_tbl, g32, err);
  else if (kind == MOE_ACT_SITU)
    act_quant_kernel<kLive, 2><<<grid, kThreads, 0, st>>>(gateup, out, out_sf, ends, E, A, M_alloc, I, ld, limit,
                                                        silu_tbl, situ_tbl, g32, err);
  else
    act_quant_kernel<kLive, 0><<<grid, kThreads, 0, st>>>(gateup, out, out_sf, ends, E, A, M_alloc, I, ld, limit,
                                                        silu_tbl, situ_tbl, g32, err);
  return cudaGetLastError();
}

// Entry i = spec_silu of the bf16 value with bits i.
__global__ void silu_table_kernel(float* __restrict__ tbl) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 65536) tbl[i] = spec_silu(bf16_to_f32((uint16_t)i));
}

// Entries i and 65536 + i: SiTU gate' and up' of the bf16 value with bits i.
__global__ void situ_table_kernel(float* __restrict__ tbl, float beta_s, float beta_l) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 65536) {
    const float v = bf16_to_f32((uint16_t)i);
    tbl[i] = spec_situ_gate(v, beta_s);
    tbl[65536 + i] = spec_situ_up(v, beta_l);
  }
}

}  // namespace

// Grid: the (x, y) plane of each expert holds gy blocks of 8 warps. gy is
// chosen from the sizes only (never from the counts), so the launch can be
// captured once and replayed: about 4 blocks per SM in total when the rows
// are spread over the experts, at least 2 per expert.
cudaError_t launch_silu_table(float* tbl, cudaStream_t st) {
  silu_table_kernel<<<256, 256, 0, st>>>(tbl);
  return cudaGetLastError();
}

cudaError_t launch_situ_table(float* tbl, float beta_s, float beta_l, cudaStream_t st) {
  situ_table_kernel<<<256, 256, 0, st>>>(tbl, beta_s, beta_l);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t* gateup, uint8_t* out, int32_t* out_sf,
                             const int32_t* expert_ends, int E, int A, int M_alloc, int I, int kind,
                             float limit, const float* silu_tbl, const float* situ_tbl, int group, int num_sms,
                             uint32_t* err, cudaStream_t st) {
  const bool g32 = group == 32;
  if (M_alloc == 0) return cudaSuccess;
  if (expert_ends) {
    if (E == 0) return cudaSuccess;
    const int gy = (int)lmin(lmax(2, (4L * num_sms + E - 1) / E), 65535);
    return launch_kind<true>(gateup, out, out_sf, expert_ends, E, A, M_alloc, I, kind, limit, silu_tbl, situ_tbl,
                             g32, dim3(1, gy, E), err, st);
  }
  const long items = (long)M_alloc * (((I / 128) + 3) / 4);
  const int gy = (int)lmin((items + 7) / 8, 8L * num_sms);
  return launch_kind<false>(gateup, out, out_sf, nullptr, 0, A, M_alloc, I, kind, limit, silu_tbl, situ_tbl,
                            g32, dim3(1, gy, 1), err, st);
}

}  // namespace moe
