// decode.cu -- sparse decode path ([SD] §3): per (token, slot) GEMVs that
// read topk_ids on the device and address only the selected expert's weights,
// the GLU between them and the weighted sum over local slots.
//
// Tensor-core path (T <= 8 tokens; the gpt-oss-shaped workload): three
// launches --
//   tc_gemv_kernel (GLU)  y1 = W_gu x + b and act = GLU(y1), per local slot
//   tc_gemv_kernel        y2 = W_d act + b, per local slot
//   weighted_sum_kernel   out = slot-ordered sum of topk_w * y2
// Each tile of 16 weight rows of a distinct selected expert is read once and
// multiplied against all token columns on the tensor cores (mma.sync
// m16n8k16); experts no slot selected, or not local, are never read ([SD]
// §3). Other shapes take four plain launches: GEMV (grid (ceil(N/32), k, T),
// a block returns block-uniformly when its slot is not local), GLU, GEMV,
// weighted sum.
//
// In the plain GEMV the activation row is staged to shared memory as fp32 with an
// XOR swizzle on 16-byte slots so that the per-lane float4 reads are free of
// bank conflicts. Each lane streams 16-byte weight chunks (16 e4m3 codes, or
// 32 e2m1 nibbles = one MXFP4 group with its UE8M0 scale) of 4 rows at once:
// 512 contiguous bytes per warp and row, coalesced.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "pipeline.cuh"

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
  pdl_wait();
  pdl_launch_dependents();  // a dependent kernel waits for this grid before reading `out`
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

// ------------------------------------------------------ tensor-core path
// For T <= 8 tokens the two GEMVs are skinny GEMMs: [16 weight rows] x [K] x
// [8 token columns]. One CTA per SM walks a contiguous range of tiles; a tile
// is 16 rows of one distinct local expert, so every selected expert's weights
// are read once however many tokens chose it. Warp 16 is the producer: its
// lanes 0-15 bulk-copy the tile's rows, one each, and lane 0 the bias (and
// MXFP4 scale bytes), into a ring of shared-memory stages. Warps 0-15 split
// K: each converts its weight slices in registers (e4m3x2 / e2m1x2 -> f16x2,
// exact) and runs mma.sync m16n8k16 (f16 x f16 -> f32) against the token
// columns, staged as f16 scaled per token by a power of two so that no bf16
// value overflows or loses bits in f16, and leaves its partial tile in one of
// kTcRedBufs reduction buffers. Warps 17-20 sum the sixteen partial tiles in
// warp order, scale them back and write every (token, slot) that selected the
// expert (the first launch applies the GLU to its gate/up row pairs on the
// way out) while the compute warps go on with the next tile. Each buffer b
// is handed over through its own pair of named barriers, 2 + b (partials
// written: the compute warps arrive, the epilogue warps wait) and
// 2 + kTcRedBufs + b (buffer free again: the other way round), so a barrier
// never has two generations in flight.
constexpr int kTcRows = 16;       // MMA M: weight rows per tile / stage
constexpr int kTcTok = 8;         // MMA N: token columns
constexpr int kTcConsumers = 16;  // warps splitting K
constexpr int kTcEpiWarps = 4;    // warps summing the partial tiles and storing the outputs
constexpr int kTcThreads = (kTcConsumers + 1 + kTcEpiWarps) * 32;
constexpr int kTcBarThreads = (kTcConsumers + kTcEpiWarps) * 32;  // compute + epilogue warps
constexpr int kTcRedBufs = 3;     // reduction buffers between the compute and epilogue warps
constexpr int kTcMaxStages = 8;
constexpr int kTcMaxSlots = 256;  // T * k
// dynamic shared memory: 227 KB per block less the kernel's static arrays
constexpr size_t kTcSmemMax = 222 * 1024;

struct TcArgs {
  const uint16_t* x;      // x [T][K] (per_slot = 0) or act [T*k][K] (per_slot = 1)
  int per_slot;
  const int32_t* ids;
  int T, k, expert_start, n_local;
  const uint8_t* W;       // [n_local][N][row_bytes]
  const float* wscale;    // FP8: [n_local]
  const uint8_t* wsf;     // MXFP4: [n_local][N][K/32]
  const uint16_t* bias;   // [n_local][N]
  int N, K;
  int glu, I, interleaved;
  float alpha, beta, limit;
  uint16_t* y;            // [slot][N]
  uint16_t* act;          // [slot][I] (glu)
  int nst;
  uint32_t stage_bytes, row_stride, sf_offset, bias_offset, x_stride;
  uint32_t* err;
};

// Source row (within the expert) of stage row r of tile q. GLU launch: stage
// rows 0-7 are the gate rows and 8-15 the up rows of intermediate indices
// 8q..8q+7, whatever the layout, so that one thread holds both halves.
__device__ __forceinline__ int tc_src_row(const TcArgs& a, int q, int r) {
  if (!a.glu) return kTcRows * q + r;
  const int i = 8 * q + (r & 7);
  if (a.interleaved) return 2 * i + (r >> 3);
  return (r < 8) ? i : a.I + i;
}
// Row, within the tile's scale and bias blocks (copied in source order), of
// stage row r.
__device__ __forceinline__ int tc_blk_row(const TcArgs& a, int r) {
  if (a.glu && a.interleaved) return 2 * (r & 7) + (r >> 3);
  return r;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(two & 0xFFFFu)));
  return h2;
}
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h2;
  asm("{.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(h2) : "h"((uint16_t)(byte & 0xFFu)));
  return h2;
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int WFMT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemv_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int K = a.K, N = a.N, nst = a.nst;
  // token columns: min(T, 8) of them; MMA columns >= T read column T - 1
  // (their outputs are never written), so the buffer is sized by T
  const int xcols = a.T < kTcTok ? a.T : kTcTok;
  uint8_t* xs = smem;                                                      // [xcols][x_stride] f16 columns
  float* red = reinterpret_cast<float*>(smem + (size_t)xcols * a.x_stride);  // [kTcRedBufs][warps][128]
  uint8_t* stages = reinterpret_cast<uint8_t*>(red + kTcRedBufs * kTcConsumers * 128);
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + (size_t)nst * a.stage_bytes);  // full[nst], empty[nst]
  __shared__ int uniq[kTcMaxSlots];
  __shared__ int ids_s[kTcMaxSlots];
  __shared__ signed char slot_tab[kTcMaxSlots][kTcTok];  // slot - t*k of token t for expert u, or -1
  __shared__ int n_uniq;
  __shared__ int warp_cnt[kTcThreads / 32];
  __shared__ int xexp[kTcTok];
  __shared__ float wmax[kTcConsumers][kTcTok];  // per-compute-warp max |x| of each column
  __shared__ float tile_sc[kTcRedBufs][kTcTok];          // per reduction buffer: column scales 2^xexp * weight scale
  __shared__ uint16_t tile_bias[kTcRedBufs][kTcRows];    // per reduction buffer: the tile's bias, source order
  __shared__ float wsc;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row_bytes = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? (size_t)K : (size_t)K / 2;
  const int sf_row = K / 32;
  const int TK = a.T * a.k;
  // The first launch may read routing, token rows or weights that the kernel
  // before it on the stream wrote, so it waits for that kernel before it reads
  // anything, and only then lets the second GEMV be scheduled (which reads the
  // routing ids before its own wait, and the first launch's activations after
  // it). The weighted sum waits for the second launch before reading y2.
  if (!a.per_slot) pdl_wait();
  pdl_launch_dependents();

  const int words = K / 2;
  // Raw bf16 pairs of token column c from activation row src (-1: not used)
  // into the column buffer, by threads [tid0, tid0 + nthr); each warp's max
  // |x| per column goes to wmax[warp][c]. Columns of tokens that did not
  // choose the expert are left stale: their outputs are never written, and
  // each MMA output column depends on its own input column only.
  auto stage_load = [&](const int (&src)[kTcTok], int nthr) {
#pragma unroll
    for (int c = 0; c < kTcTok; ++c) {
      float m = 0.0f;
      if (src[c] >= 0) {
        const uint32_t* gx = reinterpret_cast<const uint32_t*>(a.x + (size_t)src[c] * K);
        uint32_t* cell = reinterpret_cast<uint32_t*>(xs + (size_t)c * a.x_stride);
#pragma unroll 4
        for (int w = threadIdx.x; w < words; w += nthr) {
          const uint32_t p = __ldg(gx + w);
          cell[w] = p;
          m = fmaxf(m, fmaxf(fabsf(bf16_lo(p)), fabsf(bf16_hi(p))));
        }
      }
      m = warp_max_xor(m, 5);
      if (lane == 0) wmax[warp][c] = m;
    }
  };
  // f16 conversion in place, x * 2^-e with e chosen per column so that the
  // largest |x| lands in [2^14, 2^15): no f16 overflow; xexp[c] = e.
  auto stage_convert = [&](const int (&src)[kTcTok], int nwarps, int nthr) {
#pragma unroll
    for (int c = 0; c < kTcTok; ++c) {
      if (src[c] < 0) continue;
      float m = 0.0f;
      for (int w = 0; w < nwarps; ++w) m = fmaxf(m, wmax[w][c]);
      const int ex = (m > 0.0f && m <= 3.0e38f) ? ilogbf(m) - 14 : 0;
      if (threadIdx.x == 0) xexp[c] = ex;
      const float sc = pow2_f32(-ex);
      uint32_t* cell = reinterpret_cast<uint32_t*>(xs + (size_t)c * a.x_stride);
      for (int w = threadIdx.x; w < words; w += nthr) {
        const uint32_t p = cell[w];
        const __half2 hv = __floats2half2_rn(__fmul_rn(bf16_lo(p), sc), __fmul_rn(bf16_hi(p), sc));
        cell[w] = *reinterpret_cast<const uint32_t*>(&hv);
      }
    }
  };
  int tok_src[kTcTok];  // first launch: column c is token c's input row
#pragma unroll
  for (int c = 0; c < kTcTok; ++c) tok_src[c] = (!a.per_slot && c < a.T) ? c : -1;

  // Routing ids, then the distinct local experts in order of first appearance
  // (the producer can start as soon as these are known).
  {
    if ((int)threadIdx.x < TK) ids_s[threadIdx.x] = a.ids[threadIdx.x];
    if (threadIdx.x == 0) {
      abort_flag = 0;
      for (int s2 = 0; s2 < nst; ++s2) {
        pipe_mbar_init(smem_addr(bars + s2), 1);
        pipe_mbar_init(smem_addr(bars + nst + s2), kTcConsumers);  // one arrive per compute warp
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    bool first = false;
    int e = -1;
    if ((int)threadIdx.x < TK) {
      e = ids_s[threadIdx.x];
      const int lid = e - a.expert_start;
      first = lid >= 0 && lid < a.n_local;
      for (int s2 = 0; first && s2 < (int)threadIdx.x; ++s2) first = ids_s[s2] != e;
    }
    const unsigned bal = __ballot_sync(kFull, first);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    if (first) uniq[before + __popc(bal & ((1u << lane) - 1u))] = e - a.expert_start;
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < kTcThreads / 32; ++w) tot += warp_cnt[w];
      n_uniq = tot;
    }
    __syncthreads();
  }
  const int tps = N / kTcRows;
  const long total = (long)n_uniq * tps;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);

  if (warp == kTcConsumers) {
    // ------------------------------------------------------------ producer
    // Lane r < 16 copies stage row r (the rows' copies are issued in
    // parallel); lane 0 also arms the stage and copies its bias and scales.
    {
      int n = 0;
      for (int tile = t_begin; tile < t_end; ++tile, ++n) {
        const int lid = uniq[tile / tps], q = tile % tps;
        const int s = n % nst;
        int okw = 1;
        if (lane == 0 && n >= nst) okw = pipe_wait(smem_addr(bars + nst + s), ((n / nst) & 1) ^ 1, abort_v, a.err);
        if (!__shfl_sync(kFull, okw, 0)) break;
        const uint32_t full = smem_addr(bars + s);
        uint8_t* st = stages + (size_t)s * a.stage_bytes;
        const uint8_t* wexp = a.W + (size_t)lid * N * row_bytes;
        const uint16_t* bexp = a.bias + (size_t)lid * N;
        const uint32_t sf_bytes = (WFMT == MOE_WFMT_MXFP4_G32) ? (uint32_t)(kTcRows * sf_row) : 0u;
        if (lane == 0) pipe_mbar_expect_tx(full, (uint32_t)(kTcRows * row_bytes) + sf_bytes + kTcRows * 2);
        __syncwarp();
        if (lane < kTcRows)
          pipe_bulk_load(smem_addr(st + (size_t)lane * a.row_stride), wexp + (size_t)tc_src_row(a, q, lane) * row_bytes,
                         (uint32_t)row_bytes, full);
        if (lane != 0) continue;
        const bool halves = a.glu && !a.interleaved;
        const int run0 = halves ? 8 * q : kTcRows * q;  // first source row of each block run
        const int run1 = halves ? a.I + 8 * q : 0;
        const int rows = halves ? 8 : kTcRows;
        pipe_bulk_load(smem_addr(st + a.bias_offset), bexp + run0, (uint32_t)(rows * 2), full);
        if (halves) pipe_bulk_load(smem_addr(st + a.bias_offset + 16), bexp + run1, 16u, full);
        if (WFMT == MOE_WFMT_MXFP4_G32) {
          const uint8_t* sexp = a.wsf + (size_t)lid * N * sf_row;
          pipe_bulk_load(smem_addr(st + a.sf_offset), sexp + (size_t)run0 * sf_row, (uint32_t)(rows * sf_row), full);
          if (halves)
            pipe_bulk_load(smem_addr(st + a.sf_offset + 8 * sf_row), sexp + (size_t)run1 * sf_row,
                           (uint32_t)(8 * sf_row), full);
        }
      }
      n = __shfl_sync(kFull, n, 0);
      if (lane == 0)
        for (int m = (n > nst ? n - nst : 0); m < n; ++m)
          pipe_wait(smem_addr(bars + (m % nst)), (m / nst) & 1, abort_v, a.err, false);
    }
    return;
  }

  if (warp > kTcConsumers) {
    // ------------------------------------------------------------ epilogue
    // Thread i < nout owns one output pair (GLU: the gate and up row of one
    // intermediate index, one column) or one output (row, column) of the
    // 16 x 8 tile.
    const int et = (int)threadIdx.x - (kTcConsumers + 1) * 32;
    const int nout = a.glu ? 64 : 128;
    const int o_l = a.glu ? (et >> 1) : (et >> 2);
    const int o_c = a.glu ? (et & 1) : (et & 3);
    const int gl = o_l >> 2;
    const int col = 2 * (o_l & 3) + (o_c & 1);
    const int r_out = a.glu ? gl : gl + 8 * (o_c >> 1);  // stage row of the (first) output
    int n = 0;
    for (int tile = t_begin; tile < t_end; ++tile, ++n) {
      const int b = n % kTcRedBufs, u = tile / tps, q = tile % tps;
      named_barrier(2 + b, kTcBarThreads);  // the compute warps have written tile n's buffer
      const float* rb = red + (size_t)b * kTcConsumers * 128;
      const int j = (et < nout && col < a.T) ? slot_tab[u][col] : -1;
      if (j >= 0 && !*abort_v) {
        const int sl = col * a.k + j;
        const float sc = tile_sc[b][col];
        const float bias0 = bf16_to_f32(tile_bias[b][tc_blk_row(a, r_out)]);
        if (a.glu) {
          const float bias1 = bf16_to_f32(tile_bias[b][tc_blk_row(a, gl + 8)]);
          float v0 = 0.0f, v1 = 0.0f;
#pragma unroll
          for (int w = 0; w < kTcConsumers; ++w) {
            v0 += rb[w * 128 + o_l * 4 + o_c];
            v1 += rb[w * 128 + o_l * 4 + 2 + o_c];
          }
          const int r0 = tc_src_row(a, q, gl), r1 = tc_src_row(a, q, gl + 8);
          const uint16_t y0 = (uint16_t)f32_to_bf16_bits(fmaf(v0, sc, bias0));
          const uint16_t y1 = (uint16_t)f32_to_bf16_bits(fmaf(v1, sc, bias1));
          a.y[(size_t)sl * N + r0] = y0;
          a.y[(size_t)sl * N + r1] = y1;
          a.act[(size_t)sl * a.I + 8 * q + gl] =
              (uint16_t)f32_to_bf16_bits(glu_value(bf16_to_f32(y0), bf16_to_f32(y1), a.alpha, a.beta, a.limit));
        } else {
          float v = 0.0f;
#pragma unroll
          for (int w = 0; w < kTcConsumers; ++w) v += rb[w * 128 + o_l * 4 + o_c];
          a.y[(size_t)sl * N + tc_src_row(a, q, r_out)] = (uint16_t)f32_to_bf16_bits(fmaf(v, sc, bias0));
        }
      }
      named_barrier_arrive(2 + kTcRedBufs + b, kTcBarThreads);  // buffer b is free again
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int kCT = kTcConsumers * 32;
  // slot table: token t's slot j (if any) that chose expert u
  for (int idx = threadIdx.x; idx < n_uniq * kTcTok; idx += kCT) {
    const int u = idx / kTcTok, t = idx % kTcTok;
    int sl = -1;
    if (t < a.T)
      for (int j = 0; j < a.k; ++j)
        if (ids_s[t * a.k + j] - a.expert_start == uniq[u]) {
          sl = j;
          break;
        }
    slot_tab[u][t] = (signed char)sl;
  }
  if (!a.per_slot) {  // first launch: the token rows, staged once
    stage_load(tok_src, kCT);
    named_barrier(1, kCT);
    stage_convert(tok_src, kTcConsumers, kCT);
  }
  named_barrier(1, kCT);
  const int g = lane >> 2, tig = lane & 3;
  int cur_u = -1;
  bool ok = true;
  int n = 0;
  for (int tile = t_begin; tile < t_end; ++tile, ++n) {
    const int u = tile / tps;
    const int lid = uniq[u];
    if (u != cur_u) {
      // New expert: the f16 token columns (once, or per expert when the
      // columns are the slots' own activation rows) with their exponents.
      named_barrier(1, kCT);  // every compute warp is done with the previous expert's columns
      if (a.per_slot) {
        // the columns are the activation rows of the slots that chose the
        // expert: the previous kernel's output
        if (cur_u < 0) pdl_wait();
        int src[kTcTok];
#pragma unroll
        for (int c = 0; c < kTcTok; ++c) src[c] = (c < a.T && slot_tab[u][c] >= 0) ? c * a.k + slot_tab[u][c] : -1;
        stage_load(src, kCT);
        named_barrier(1, kCT);
        stage_convert(src, kTcConsumers, kCT);
      }
      if (threadIdx.x == 0) wsc = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? a.wscale[lid] : 1.0f;
      named_barrier(1, kCT);
      cur_u = u;
    }
    const int s = n % nst;
    if (ok) ok = pipe_wait(smem_addr(bars + s), (n / nst) & 1, abort_v, a.err);
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint8_t* st = stages + (size_t)s * a.stage_bytes;
    if (ok) {
      const uint8_t* rowA = st + (size_t)g * a.row_stride;
      const uint8_t* rowB = st + (size_t)(g + 8) * a.row_stride;
      const uint8_t* xg = xs + (size_t)(g < xcols ? g : xcols - 1) * a.x_stride;
      if (WFMT == MOE_WFMT_FP8_PER_EXPERT) {
        float d2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2  // two k-blocks' loads and conversions in flight: 3-4% faster than one
        for (int kb = warp; kb < K / 64; kb += kTcConsumers) {
          const int k0 = kb * 64 + 16 * tig;
          const uint4 wa = *reinterpret_cast<const uint4*>(rowA + k0);
          const uint4 wb = *reinterpret_cast<const uint4*>(rowB + k0);
          const uint4 x0 = *reinterpret_cast<const uint4*>(xg + 2 * k0);
          const uint4 x1 = *reinterpret_cast<const uint4*>(xg + 2 * k0 + 16);
          mma_f16(d, e4m3x2_to_f16x2(wa.x), e4m3x2_to_f16x2(wb.x), e4m3x2_to_f16x2(wa.x >> 16),
                  e4m3x2_to_f16x2(wb.x >> 16), x0.x, x0.y);
          mma_f16(d2, e4m3x2_to_f16x2(wa.y), e4m3x2_to_f16x2(wb.y), e4m3x2_to_f16x2(wa.y >> 16),
                  e4m3x2_to_f16x2(wb.y >> 16), x0.z, x0.w);
          mma_f16(d, e4m3x2_to_f16x2(wa.z), e4m3x2_to_f16x2(wb.z), e4m3x2_to_f16x2(wa.z >> 16),
                  e4m3x2_to_f16x2(wb.z >> 16), x1.x, x1.y);
          mma_f16(d2, e4m3x2_to_f16x2(wa.w), e4m3x2_to_f16x2(wb.w), e4m3x2_to_f16x2(wa.w >> 16),
                  e4m3x2_to_f16x2(wb.w >> 16), x1.z, x1.w);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += d2[i];
      } else {
        const uint8_t* sfs = st + a.sf_offset;
        const uint8_t* sfA = sfs + (size_t)tc_blk_row(a, g) * sf_row;
        const uint8_t* sfB = sfs + (size_t)tc_blk_row(a, g + 8) * sf_row;
#pragma unroll 3  // three groups in flight (1-2% faster than one or two)
        for (int grp = warp; grp < sf_row; grp += kTcConsumers) {
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(rowA + 16 * grp + 4 * tig);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(rowB + 16 * grp + 4 * tig);
          const uint4 xv = *reinterpret_cast<const uint4*>(xg + 2 * (32 * grp + 8 * tig));
          // both halves of the 32-wide scale group accumulate in one fragment
          float e1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma_f16(e1, e2m1x2_to_f16x2(wa), e2m1x2_to_f16x2(wb), e2m1x2_to_f16x2(wa >> 8), e2m1x2_to_f16x2(wb >> 8),
                  xv.x, xv.y);
          mma_f16(e1, e2m1x2_to_f16x2(wa >> 16), e2m1x2_to_f16x2(wb >> 16), e2m1x2_to_f16x2(wa >> 24),
                  e2m1x2_to_f16x2(wb >> 24), xv.z, xv.w);
          const float sA = pow2_f32((int)sfA[grp] - 127), sB = pow2_f32((int)sfB[grp] - 127);
          d[0] = fmaf(e1[0], sA, d[0]);
          d[1] = fmaf(e1[1], sA, d[1]);
          d[2] = fmaf(e1[2], sB, d[2]);
          d[3] = fmaf(e1[3], sB, d[3]);
        }
      }
    }
    // Warp 0 takes the tile's bias out of the stage; each compute warp
    // releases the stage when it is done with it (its generic-proxy reads
    // fenced before the next bulk copy refills the stage): the stage's empty
    // barrier completes once all sixteen have.
    uint16_t bias_v = 0;
    if (warp == 0 && lane < kTcRows && ok) bias_v = reinterpret_cast<const uint16_t*>(st + a.bias_offset)[lane];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0 && ok) pipe_mbar_arrive(smem_addr(bars + nst + s));
    // The partial tile, the bias and the column scales into reduction buffer
    // b, free once the epilogue warps are done with tile n - kTcRedBufs.
    const int b = n % kTcRedBufs;
    if (n >= kTcRedBufs) named_barrier(2 + kTcRedBufs + b, kTcBarThreads);
    float* rb = red + (size_t)b * kTcConsumers * 128;
    *reinterpret_cast<float4*>(rb + warp * 128 + lane * 4) = make_float4(d[0], d[1], d[2], d[3]);
    if (warp == 0) {
      if (lane < kTcRows) tile_bias[b][lane] = bias_v;
      if (lane < kTcTok) tile_sc[b][lane] = lane < a.T ? pow2_f32(xexp[lane]) * wsc : 0.0f;
    }
    named_barrier_arrive(2 + b, kTcBarThreads);  // tile n to the epilogue warps
  }
  // the epilogue warps' releases of the last buffers
  for (int m = (n > kTcRedBufs ? n - kTcRedBufs : 0); m < n; ++m)
    named_barrier(2 + kTcRedBufs + m % kTcRedBufs, kTcBarThreads);
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

cudaError_t launch_weighted_sum(const moe_decode_args& a, bool pdl, cudaStream_t st) {
  const long total = (long)a.T * a.H;
  return launch_maybe_pdl(weighted_sum_kernel, dim3((int)lmin((total + 255) / 256, 4096)), dim3(256), 0, st, pdl,
                          (const uint16_t*)a.y2, a.topk_ids, a.topk_w, a.T, a.k, a.expert_start,
                          a.num_local_experts, a.H, a.out);
}

// Shared-memory geometry of the tensor-core path. Row strides are padded so
// that the warp's 16-byte (FP8) or 4-byte (MXFP4) weight loads and its
// 16-byte token-column loads hit distinct banks.
struct TcGeom {
  uint32_t row_stride, sf_offset, bias_offset, stage_bytes, x_stride;
  int nst;
  size_t smem;
};

static uint32_t pad_to(uint32_t v, uint32_t residue) {  // smallest >= v with v % 128 == residue
  return v + ((residue + 128u - v % 128u) % 128u);
}

template <int WFMT>
TcGeom tc_geom(int K, int T) {
  const size_t xcols = (size_t)(T < kTcTok ? (T > 1 ? T : 1) : kTcTok);
  TcGeom g{};
  const uint32_t rb = (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? (uint32_t)K : (uint32_t)K / 2;
  g.row_stride = pad_to(rb, (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? 64u : 16u);
  g.sf_offset = kTcRows * g.row_stride;
  const uint32_t sf = (WFMT == MOE_WFMT_MXFP4_G32) ? (uint32_t)(kTcRows * (K / 32)) : 0u;
  g.bias_offset = (g.sf_offset + sf + 15u) / 16u * 16u;
  g.stage_bytes = (g.bias_offset + kTcRows * 2 + 127u) / 128u * 128u;
  g.x_stride = pad_to(2u * (uint32_t)K, (WFMT == MOE_WFMT_FP8_PER_EXPERT) ? 16u : 64u);
  const size_t fixed = xcols * g.x_stride + kTcRedBufs * kTcConsumers * 128 * sizeof(float) +
                       2 * kTcMaxStages * sizeof(uint64_t);
  g.nst = 0;
  if (fixed < kTcSmemMax) {
    const size_t n = (kTcSmemMax - fixed) / g.stage_bytes;
    g.nst = (int)(n < (size_t)kTcMaxStages ? n : (size_t)kTcMaxStages);
  }
  g.smem = xcols * g.x_stride + kTcRedBufs * kTcConsumers * 128 * sizeof(float) + (size_t)g.nst * g.stage_bytes +
           2 * (size_t)g.nst * sizeof(uint64_t);
  return g;
}

// The tensor-core path takes T <= 8, T * k <= 256, N % 16 == 0, K % 64 == 0
// (FP8: 64-wide K blocks; MXFP4: 8-row scale runs stay 16-byte multiples) and
// at least two stages.
template <int WFMT>
bool tc_ok(int T, int k, int N, int K) {
  return T <= kTcTok && T * k <= kTcMaxSlots && N % kTcRows == 0 && K % 64 == 0 && tc_geom<WFMT>(K, T).nst >= 2;
}

template <int WFMT>
cudaError_t launch_tc(TcArgs s, int num_sms, cudaStream_t st, bool pdl) {
  const TcGeom g = tc_geom<WFMT>(s.K, s.T);
  s.nst = g.nst;
  s.stage_bytes = g.stage_bytes;
  s.row_stride = g.row_stride;
  s.sf_offset = g.sf_offset;
  s.bias_offset = g.bias_offset;
  s.x_stride = g.x_stride;
  // tiles = distinct experts (at most min(T*k, n_local)) x N/16; the grid is
  // fixed by the sizes so that a captured graph replays under new routing
  const long max_tiles = lmin((long)s.T * s.k, (long)s.n_local) * (s.N / kTcRows);
  const int grid = (int)lmin(max_tiles, (long)num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_maybe_pdl(tc_gemv_kernel<WFMT>, dim3(grid), dim3(kTcThreads), g.smem, st, pdl, s);
}

template <int WFMT>
cudaError_t launch_decode_tc(const moe_decode_args& a, const float* gu_scale, const uint8_t* gu_sf,
                             const float* d_scale, const uint8_t* d_sf, int num_sms, uint32_t* err, cudaStream_t st) {
  TcArgs s{};
  s.ids = a.topk_ids;
  s.T = a.T;
  s.k = a.k;
  s.expert_start = a.expert_start;
  s.n_local = a.num_local_experts;
  s.err = err;
  // GEMV 1 + GLU
  s.x = a.x;
  s.per_slot = 0;
  s.W = a.w_gu;
  s.wscale = gu_scale;
  s.wsf = gu_sf;
  s.bias = a.b_gu;
  s.N = 2 * a.I;
  s.K = a.H;
  s.glu = 1;
  s.I = a.I;
  s.interleaved = a.glu_layout == MOE_GLU_INTERLEAVED;
  s.alpha = a.glu_alpha;
  s.beta = a.glu_beta;
  s.limit = a.glu_limit;
  s.y = a.y1;
  s.act = a.act;
  cudaError_t ce = launch_tc<WFMT>(s, num_sms, st, true);
  if (ce != cudaSuccess) return ce;
  // GEMV 2
  s.x = a.act;
  s.per_slot = 1;
  s.W = a.w_d;
  s.wscale = d_scale;
  s.wsf = d_sf;
  s.bias = a.b_d;
  s.N = a.H;
  s.K = a.I;
  s.glu = 0;
  s.y = a.y2;
  s.act = nullptr;
  if ((ce = launch_tc<WFMT>(s, num_sms, st, true)) != cudaSuccess) return ce;
  return launch_weighted_sum(a, true, st);
}

cudaError_t init_decode() {
  cudaError_t ce;
  if ((ce = cudaFuncSetAttribute(tc_gemv_kernel<MOE_WFMT_FP8_PER_EXPERT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kTcSmemMax)) != cudaSuccess)
    return ce;
  return cudaFuncSetAttribute(tc_gemv_kernel<MOE_WFMT_MXFP4_G32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kTcSmemMax);
}

bool decode_mma_sync_ok(const moe_decode_args& a) {
  if (a.wfmt == MOE_WFMT_FP8_PER_EXPERT)
    return tc_ok<MOE_WFMT_FP8_PER_EXPERT>(a.T, a.k, 2 * a.I, a.H) && tc_ok<MOE_WFMT_FP8_PER_EXPERT>(a.T, a.k, a.H, a.I);
  return tc_ok<MOE_WFMT_MXFP4_G32>(a.T, a.k, 2 * a.I, a.H) && tc_ok<MOE_WFMT_MXFP4_G32>(a.T, a.k, a.H, a.I);
}

cudaError_t launch_decode(const moe_decode_args& a, bool allow_mma_sync, int num_sms, uint32_t* err,
                          cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t ce;
  const bool fp8 = a.wfmt == MOE_WFMT_FP8_PER_EXPERT;
  if (allow_mma_sync && decode_mma_sync_ok(a))
    return fp8 ? launch_decode_tc<MOE_WFMT_FP8_PER_EXPERT>(a, a.w_gu_scale, nullptr, a.w_d_scale, nullptr, num_sms, err,
                                                           st)
               : launch_decode_tc<MOE_WFMT_MXFP4_G32>(a, nullptr, a.w_gu_sf, nullptr, a.w_d_sf, num_sms, err, st);
  // Otherwise four launches: GEMV, GLU, GEMV, weighted sum.
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
  return launch_weighted_sum(a, false, st);
}

}  // namespace moe
