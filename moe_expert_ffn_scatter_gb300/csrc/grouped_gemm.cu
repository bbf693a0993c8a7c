// grouped_gemm.cu -- block-scaled grouped GEMM over live rows on the sm_103a
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
//   out[r, n] = bf16( sum_k e4m3(a[r,k]) 2^(sa(r, k/128) - 127)
//                           * w(e, n, k) 2^(sw(e, n, k/32) - 127) )
// for the live rows r in [start[e], end[e]) of every expert e; A = 128-row
// aligned segments ([LR] §2: FC1 and FC2 take the same endpoint layout, and
// padding rows are never computed; [DG] §2.3.1 recipes (1,128) activations,
// (1,32) MXFP4 weights).
//
// Kernel structure (one persistent CTA per SM, 256 threads):
//   warp 0    TMA producer: 128x128 e4m3 A tile and 256x128 B tile per stage
//             (B e2m1 is expanded by TMA to one byte per element, the layout
//             kind::mxf8f6f4 reads for 4-bit operands; the transaction count
//             of such a copy is its packed global size), 128B swizzle.
//   warp 1    TMEM owner and MMA issuer: tcgen05.cp moves the stage's scale
//             factors from shared to tensor memory, then 4 x
//             tcgen05.mma.kind::mxf8f6f4.block_scale (M128 N256 K32) into a
//             128x256 fp32 accumulator; tcgen05.commit frees the stage.
//             The same thread bulk-copies the stage's scale words: the
//             activation scales (one int32 holds 4 groups of 128 of the packed
//             MN-major array, used as stored: the MMA's scale-factor-A id
//             picks the byte) and the prepared weight scales (4 x 32-K blocks
//             per int32, picked by the scale-factor-B id, pre-permuted at load
//             time into the 32-row x 16-byte source layout of tcgen05.cp
//             32x128b.warpx4).
//   warp 2    activation-scale transposer: rearranges the 128 activation scale
//             words of each stage into that tcgen05.cp source layout
//             (shared -> shared), then completes the stage's full barrier.
//   warps 4-7 epilogue: tcgen05.ld of the accumulator (each warp its 32-lane
//             quarter), bf16 conversion into registers, accumulator released;
//             then (GEMM1 fused) SiLU from a shared-memory window of the table,
//             times up, and the e4m3/UE8M0 quantisation; the rows go out through
//             a 2 KB per-warp shared buffer, 64 contiguous bytes of 8 rows per
//             store instruction (rows >= end[e] are skipped).
// The tile list is (live 128-row tile, 256-column tile); the number of live
// tiles, align_up(end[E-1], 128) / 128, and each tile's expert come from the
// device-side endpoint tensor, so the grid never depends on routing counts.
// Every mbarrier wait is bounded (about one second); a wait that runs out sets
// MOE_DEVERR_WAIT_TIMEOUT, makes every role leave its loop, drains the issued
// tensor-core work and frees tensor memory before the CTA exits.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {

namespace {

#ifndef MOE_GEMM_STAGES
#define MOE_GEMM_STAGES 4
#endif
constexpr int BM = 128, BN = 256, BK = 128, STAGES = MOE_GEMM_STAGES;
constexpr int kThreads = 256;
constexpr uint32_t A_BYTES = BM * BK;
constexpr uint32_t B_BYTES = BN * BK;
constexpr uint32_t SFA_BYTES = BM * 4;
constexpr uint32_t SFB_BYTES = BN * 4;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;          // tcgen05.cp layout
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;       // tcgen05.cp layout
constexpr uint32_t OFF_SFA_IN = OFF_SFB + STAGES * SFB_BYTES;    // activation scales as stored
constexpr uint32_t OFF_BAR = OFF_SFA_IN + STAGES * SFA_BYTES;
constexpr uint32_t NUM_BARS = 3 * STAGES + 3;
constexpr uint32_t OFF_TMEM_PTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_PTR + 4;
constexpr uint32_t OFF_ENDS = OFF_ABORT + 12;                   // expert_ends copy (E <= kSmemExperts)
constexpr int kSmemExperts = 1024;
constexpr uint32_t STG_BYTES = 2048;                              // per epilogue warp: 32 rows x 64 bytes
constexpr uint32_t OFF_STG = (OFF_ENDS + kSmemExperts * 4 + 15) / 16 * 16;
// SiLU window: the table entries of the bf16 gate values with |g| in
// [2^-6, 2^6) (exponent field 121..132), positive then negative, 1536 each.
constexpr uint32_t kWinBase = 121u << 7;  // bits 0x3C80
constexpr uint32_t kWinHalf = 12u * 128u;
constexpr uint32_t OFF_WIN = OFF_STG + 4 * STG_BYTES;
constexpr uint32_t SMEM_USED = OFF_WIN + 2 * kWinHalf * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SF_BASE = 256;             // stage s: SFA cols 256+16s, SFB cols 264+16s

static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale:
// A format e4m3 (0), B format e2m1 (5) or e4m3 (0), both K-major, N >> 3 at
// bit 17, UE8M0 scale type at bit 23, M >> 4 at bit 24; the scale-factor ids
// (B at bit 4, A at bit 29) are or-ed in per instruction.
__host__ __device__ constexpr uint32_t idesc_base(bool b_fp4) {
  return (0u << 7) | ((b_fp4 ? 5u : 0u) << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
         ((uint32_t)(BM >> 4) << 24);
}

// Expert of the live 128-row tile starting at m0: the smallest e with
// align_up(end[e], 128) > m0 (start[e] <= m0 < end[e] follows). `ends` is
// the shared-memory copy of the endpoint tensor.
__device__ __forceinline__ int expert_of_tile(const int32_t* ends, int E, int m0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int)align_up64(ends[mid], BM) > m0) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// SiLU of the bf16 gate value with bits `bits` (low 16): from the shared
// window (the kWinH patterns from kWinB up, positive then negative) when |g|
// lies in it, else from the per-context table in global memory.
template <uint32_t kWinB, uint32_t kWinH>
__device__ __forceinline__ float silu_windowed(const float* win, const float* __restrict__ tbl, uint32_t bits) {
  const uint32_t b = bits & 0xFFFFu;
  const uint32_t off = (b & 0x7FFFu) - kWinB;
  if (off < kWinH) return win[off + ((b & 0x8000u) ? kWinH : 0u)];
  return __ldg(tbl + b);
}

// Stores 64 bytes of each of the warp's 32 rows: lane r holds row r's four
// 16-byte units in u, row r goes to dst + r * ld (bytes), and rows r >= nrows
// are not written. The rows pass through the warp's staging buffer so that
// each global store instruction covers 64 contiguous bytes of 8 rows, where a
// direct store from the row-per-lane layout touches 32 rows. Unit j of row r
// sits at 16 * (j ^ ((r >> 1) & 3)) in its row: the writes and the reads are
// both free of bank conflicts.
__device__ __forceinline__ void store_rows64(uint32_t stg, int lane, const uint32_t (&u)[16], uint8_t* dst,
                                             size_t ld, int nrows) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)),
                 "r"(u[4 * j]), "r"(u[4 * j + 1]), "r"(u[4 * j + 2]), "r"(u[4 * j + 3])
                 : "memory");
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2), j = lane & 3;
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(stg + r * 64 + ((j ^ ((r >> 1) & 3)) << 4))
                 : "memory");
    if (r < nrows) *reinterpret_cast<uint4*>(dst + (size_t)r * ld + 16 * j) = v;
  }
  __syncwarp();
}

// Epilogue kinds: bf16 output, or (GEMM1 with gate/up rows interleaved in
// blocks of 128) SiLU*mul + e4m3/UE8M0 quantisation of the bf16-rounded
// accumulators, optionally with the gate/up clamp, or SiTU (gate' and up'
// from the per-context tables) + the same quantisation.
constexpr int kEpiBf16 = 0, kEpiSilu = 1, kEpiSiluClamp = 2, kEpiSitu = 3;

// Epilogue of one 128 x 256 accumulator tile, for the warp holding rows
// rbase .. rbase + 31 (lane = row) in `packed` (the 256 accumulator columns
// as bf16 pairs, already read from tensor memory and released): bf16 rows
// out, or (GEMM1 with gate/up interleaved in blocks of 128) SiLU*mul +
// e4m3/UE8M0 quantisation. Rows >= row_end are not written. stg: the warp's
// 2 KB staging buffer; win: the shared SiLU window [kWinB, kWinB + kWinH)
// of exponent-field-ordered bf16 patterns, positive then negative.
template <int kEpi, uint32_t kWinB, uint32_t kWinH>
__device__ __forceinline__ void epilogue_tile(uint32_t (&packed)[BN / 2], int lane, int rbase, int row_end, int n0,
                                              int N, uint16_t* __restrict__ out, uint8_t* __restrict__ out_q,
                                              int32_t* __restrict__ out_sf, int ld_out_sf, float limit,
                                              float silu_limit, const float* win,
                                              const float* __restrict__ silu_tbl,
                                              const float* __restrict__ situ_tbl, bool out_g32, uint32_t stg) {
  const int row = rbase + lane;
  if (kEpi == kEpiBf16) {
    // 32 columns (64 bytes) of the warp's rows at a time
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t u[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = packed[16 * c + i];
      store_rows64(stg, lane, u, reinterpret_cast<uint8_t*>(out + (size_t)rbase * N + n0 + 32 * c),
                   (size_t)N * 2, row_end - rbase);
    }
  } else {
    // This thread holds its row's gate (columns 0-127) and up (128-255)
    // of one 128-column group, already rounded to bf16 like the stored
    // gate/up buffer of the unfused path; with the same SiLU table the
    // result is bitwise that of the act-quant kernel on that buffer.
    const int grp = n0 / BN;
    const int I = N / 2;
    float amax4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // per 32 columns of h
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float ga = bf16_lo(packed[i]), gb = bf16_hi(packed[i]);
      float ua = bf16_lo(packed[64 + i]), ub = bf16_hi(packed[64 + i]);
      float sa, sb;
      if (kEpi == kEpiSitu) {
        sa = __ldg(situ_tbl + (packed[i] & 0xFFFFu));
        sb = __ldg(situ_tbl + (packed[i] >> 16));
        ua = __ldg(situ_tbl + 65536 + (packed[64 + i] & 0xFFFFu));
        ub = __ldg(situ_tbl + 65536 + (packed[64 + i] >> 16));
      } else {
        if (kEpi == kEpiSiluClamp) {
          ua = fminf(fmaxf(ua, -limit), limit);
          ub = fminf(fmaxf(ub, -limit), limit);
        }
        // with the clamp, gate values above the limit (or NaN) take spec_silu(limit)
        const bool over_a = kEpi == kEpiSiluClamp && !(ga <= limit) && !isnan(limit);
        const bool over_b = kEpi == kEpiSiluClamp && !(gb <= limit) && !isnan(limit);
        sa = over_a ? silu_limit : silu_windowed<kWinB, kWinH>(win, silu_tbl, packed[i]);
        sb = over_b ? silu_limit : silu_windowed<kWinB, kWinH>(win, silu_tbl, packed[i] >> 16);
      }
      const float2 hh = mul2(make_float2(sa, sb), make_float2(ua, ub));
      packed[i] = __float_as_uint(hh.x);       // h[2i]
      packed[64 + i] = __float_as_uint(hh.y);  // h[2i + 1]
      amax4[i >> 4] = fmaxf(amax4[i >> 4], fmaxf(fabsf(hh.x), fabsf(hh.y)));
    }
    // one scale for the 128 columns, or one per 32 (MXFP8 recipe)
    uint32_t bq[4];
    if (out_g32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) bq[j] = group_scale_byte(amax4[j]);
    } else {
      const uint32_t b = group_scale_byte(fmaxf(fmaxf(amax4[0], amax4[1]), fmaxf(amax4[2], amax4[3])));
#pragma unroll
      for (int j = 0; j < 4; ++j) bq[j] = b;
    }
    // the 128 e4m3 codes of the row, 64 bytes (4 x 16 codes) at a time;
    // every lane takes part in the staging, rows past the end are not stored
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      uint32_t u[16];
#pragma unroll
      for (int vv = 0; vv < 4; ++vv) {
        const int v = 4 * hb + vv;
        const float sc = pow2_f32(127 - (int)bq[v >> 1]);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int j = 16 * v + 4 * w;  // h[j] = packed[j/2] (j even), packed[64 + j/2] (j odd)
          const float h0 = __uint_as_float(packed[j / 2]), h1 = __uint_as_float(packed[64 + j / 2]);
          const float h2 = __uint_as_float(packed[j / 2 + 1]), h3 = __uint_as_float(packed[64 + j / 2 + 1]);
          u[4 * vv + w] = e4m3x2_satfinite(__fmul_rn(h0, sc), __fmul_rn(h1, sc)) |
                          (e4m3x2_satfinite(__fmul_rn(h2, sc), __fmul_rn(h3, sc)) << 16);
        }
      }
      store_rows64(stg, lane, u, out_q + (size_t)rbase * I + (size_t)grp * 128 + 64 * hb, (size_t)I,
                   row_end - rbase);
    }
    if (row < row_end) {
      if (out_g32) {
        out_sf[(size_t)grp * ld_out_sf + row] = (int32_t)(bq[0] | (bq[1] << 8) | (bq[2] << 16) | (bq[3] << 24));
      } else {
        uint8_t* sfb = reinterpret_cast<uint8_t*>(out_sf) + ((size_t)(grp >> 2) * ld_out_sf + row) * 4;
        sfb[grp & 3] = (uint8_t)bq[0];
        const int G = I / 128;
        if (grp == G - 1)
          for (int t = (grp & 3) + 1; t < 4; ++t) sfb[t] = 0;  // unused bytes of the last word
      }
    }
  }
}

template <bool kBfp4, int kEpi>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const int32_t* __restrict__ a_sf, int ld_sf, const int32_t* __restrict__ ends, int E, int cap,
    const uint32_t* __restrict__ w_sf, int N, int K, uint16_t* __restrict__ out, uint8_t* __restrict__ out_q,
    int32_t* __restrict__ out_sf, int ld_out_sf, float limit, const float* __restrict__ silu_tbl,
    const float* __restrict__ situ_tbl, bool a_g32, bool out_g32, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_PTR);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto sfa_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t tmem_full_bar = bar0 + 8u * (3 * STAGES);
  const uint32_t tmem_empty_bar = bar0 + 8u * (3 * STAGES + 1);
  const uint32_t done_bar = bar0 + 8u * (3 * STAGES + 2);

  // The endpoints, from a shared copy when they fit, else from global memory.
  const int32_t* ends_s = ends;
  if (E <= kSmemExperts) {
    int32_t* copy = reinterpret_cast<int32_t*>(smem + OFF_ENDS);
    for (int i = threadIdx.x; i < E; i += blockDim.x) copy[i] = __ldg(ends + i);
    ends_s = copy;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 2);   // producer's expect_tx arrive + scale transposer's arrive
      mbar_init(empty_bar(s), 1);  // tcgen05.commit
      mbar_init(sfa_bar(s), 1);    // producer's expect_tx arrive for the activation scales
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, 4);  // one arrive per epilogue warp
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int KC = K / BK;
  const int n_tiles = N / BN;
  int rows_aligned = (int)align_up64(ends_s[E - 1], BM);
  if (rows_aligned > cap || rows_aligned < 0) {
    if (threadIdx.x == 0) raise_error(err, MOE_DEVERR_ENDPOINTS);
    rows_aligned = 0;
  }
  const int num_tiles = (rows_aligned / BM) * n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
      int s = 0;
      uint32_t ph = 0;
      int issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m0 = (tile / n_tiles) * BM, n0 = (tile % n_tiles) * BN;
        const int e = expert_of_tile(ends_s, E, m0);
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(empty_bar(s), ph ^ 1u, abort_flag, err))) break;
          mbar_arrive_expect_tx(sfa_bar(s), SFA_BYTES);
          // group-128 scales: word kc/4 holds the k-block's group in byte kc%4;
          // group-32 scales (MXFP8): word kc holds its four 32-K groups
          bulk_load(sbase + OFF_SFA_IN + s * SFA_BYTES, a_sf + (size_t)(a_g32 ? kc : (kc >> 2)) * ld_sf + m0,
                    SFA_BYTES, sfa_bar(s));
          mbar_arrive_expect_tx(full_bar(s), A_BYTES + (kBfp4 ? B_BYTES / 2 : B_BYTES) + SFB_BYTES);
          tma_load_2d(sbase + OFF_A + s * A_BYTES, &tmA, kc * BK, m0, full_bar(s));
          tma_load_2d(sbase + OFF_B + s * B_BYTES, &tmB, kc * BK, e * N + n0, full_bar(s));
          bulk_load(sbase + OFF_SFB + s * SFB_BYTES, w_sf + ((size_t)e * KC + kc) * N + n0, SFB_BYTES, full_bar(s));
          issued[s] = (int)ph;
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA can exit: their
        // transaction bytes complete the full barriers' tx counts whether or
        // not the scale loader arrived, so wait with a short bound only.
        for (int i = 0; i < STAGES; ++i)
          if (issued[i] >= 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(full_bar(i), (uint32_t)issued[i]) && globaltimer_ns() - t0 < 2000000ull) {}
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      const uint32_t ibase = idesc_base(kBfp4);
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!(ok = wait_phase(tmem_empty_bar, acc_ph ^ 1u, abort_flag, err))) break;
        tc_fence_after();
        for (int kc = 0; kc < KC; ++kc) {
          if (!(ok = wait_phase(full_bar(s), ph, abort_flag, err))) break;
          tc_fence_after();
          const uint32_t tsfa = tmem + TMEM_SF_BASE + 16u * s;
          const uint32_t tsfb = tsfa + 8u;
          tc_cp_sf(tsfa, desc_sf(sbase + OFF_SFA + s * SFA_BYTES));
          tc_cp_sf(tsfb, desc_sf(sbase + OFF_SFB + s * SFB_BYTES));
          tc_cp_sf(tsfb + 4u, desc_sf(sbase + OFF_SFB + s * SFB_BYTES + 512u));
          const uint32_t a_addr = sbase + OFF_A + s * A_BYTES;
          const uint32_t b_addr = sbase + OFF_B + s * B_BYTES;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t idesc = ibase | ((uint32_t)k4 << 4) | ((uint32_t)(a_g32 ? k4 : (kc & 3)) << 29);
            tc_mma(tmem, desc_sw128(a_addr + 32u * k4), desc_sw128(b_addr + 32u * k4), idesc, tsfa, tsfb,
                   (kc | k4) != 0);
          }
          tc_commit(empty_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tmem_full_bar);
        acc_ph ^= 1u;
      }
      // Drain: every tcgen05 operation issued above completes before the
      // tensor memory is released.
      tc_commit(done_bar);
      wait_phase(done_bar, 0, abort_flag, err, false);
    }
  } else if (warp == 2) {
    // ------------------------------------------- activation-scale transposer
    // The bulk copy lands the 128 scale words of the tile's rows in row order;
    // tcgen05.cp 32x128b.warpx4 wants word (i, j) of its 32 x 4 source at
    // 16 i + 4 j to hold row 32 j + i. Lane i gathers rows i, 32+i, 64+i, 96+i.
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    const int total = (num_tiles > (int)blockIdx.x) ? ((num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * KC : 0;
    for (int it = 0; it < total; ++it) {
      if (!(ok = wait_phase(sfa_bar(s), ph, abort_flag, err))) break;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(smem + OFF_SFA_IN + s * SFA_BYTES);
      uint4 v;
      v.x = src[lane];
      v.y = src[32 + lane];
      v.z = src[64 + lane];
      v.w = src[96 + lane];
      *reinterpret_cast<uint4*>(smem + OFF_SFA + s * SFA_BYTES + 16 * lane) = v;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(s));
      if (++s == STAGES) { s = 0; ph ^= 1u; }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ epilogue
    const int q = warp & 3;
    const float silu_limit = (kEpi == kEpiSiluClamp) ? spec_silu(limit) : 0.0f;
    // The epilogue warps fill the SiLU window (the single-warp-per-scheduler
    // epilogue waits out every table lookup; shared memory answers far sooner
    // than the small L1 left beside this kernel's shared memory).
    float* win = reinterpret_cast<float*>(smem + OFF_WIN);
    if (kEpi == kEpiSilu || kEpi == kEpiSiluClamp) {
      for (int i = threadIdx.x - 128; i < (int)(2 * kWinHalf); i += 128)
        win[i] = __ldg(silu_tbl + (i < (int)kWinHalf ? kWinBase + i : 0x8000u + kWinBase + (i - kWinHalf)));
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    uint32_t acc_ph = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m0 = (tile / n_tiles) * BM, n0 = (tile % n_tiles) * BN;
      const int e = expert_of_tile(ends_s, E, m0);
      const int row_end = ends_s[e];
      if (!wait_phase(tmem_full_bar, acc_ph, abort_flag, err)) break;
      tc_fence_after();
      uint32_t packed[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 32; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + 32u * c, r0);
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + 32u * (c + 1), r1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          packed[16 * c + i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
          packed[16 * (c + 1) + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty_bar);
      epilogue_tile<kEpi, kWinBase, kWinHalf>(packed, lane, m0 + 32 * q, row_end, n0, N, out, out_q, out_sf,
                                               ld_out_sf, limit, silu_limit, win, silu_tbl, situ_tbl, out_g32,
                                               sbase + OFF_STG + q * STG_BYTES);
      acc_ph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ===================================================================
// CTA-pair kernel (cta_group::2). Two CTAs of a cluster share one
// M256 x N256 tile: the even CTA holds rows [m0, m0 + 128) and weight rows
// [n0, n0 + 128) of the tile, the odd CTA rows [m0 + 128, m0 + 256) and
// weight rows [n0 + 128, n0 + 256). The even CTA's thread issues
// tcgen05.mma.cta_group::2 (M256 N256 K32): each SM multiplies its own 128
// activation rows by both weight halves into its own 128 x 256 accumulator,
// with its own activation scales and the full tile's weight scales in its own
// tensor memory (each CTA loads all 256 rows' weight scales). One pair MMA
// runs at about twice the rate per SM of the one-CTA M128 form.
//
// Pair tiles follow the endpoint layout: expert e gets ceil(count_e / 256)
// row tiles starting at start[e]; when the last one holds 128 rows or fewer,
// the odd CTA's rows lie past end[e]: it loads no activation rows (its stale
// shared memory gives rows nobody stores) but still loads its weight half.
//
// Per stage, each CTA's copies complete on its own `full` barrier; its scale
// transposer then rearranges the activation scales in place and arrives on
// the even CTA's `ready` barrier (locally or through the cluster), which the
// issuer waits for. Every wait is local and bounded; the issuer's commits
// arrive on both CTAs' `empty` / `tmem_full` barriers (multicast), and the
// epilogue warps of both CTAs release the accumulators on the even CTA's
// `tmem_empty` barrier.
namespace pr {
// A stage holds KSUB 128-wide k-blocks. Six single-k-block stages keep
// about six k-blocks of loads in flight ahead of the tensor cores; the scale
// copies are issued by CTA 0's transposer, so the issuing thread's own cost
// per stage (barrier wait, four MMAs, commit) stays within the MMAs' time.
#ifndef MOE_GEMM_PAIR_STAGES
#define MOE_GEMM_PAIR_STAGES 6
#endif
#ifndef MOE_GEMM_PAIR_KSUB
#define MOE_GEMM_PAIR_KSUB 1
#endif
constexpr int STAGES = MOE_GEMM_PAIR_STAGES;
constexpr int KSUB = MOE_GEMM_PAIR_KSUB;        // k-blocks per stage
constexpr uint32_t A_SUB = BM * BK;              // this CTA's 128 rows, one k-block
constexpr uint32_t B_SUB = (BN / 2) * BK;        // this CTA's half of the weight tile, one k-block
constexpr uint32_t SFA_SUB = BM * 4;             // activation scale words of one k-block
constexpr uint32_t SFB_SUB = BN * 4;             // the whole tile's weight scales of one k-block
constexpr uint32_t A_BYTES = KSUB * A_SUB;
constexpr uint32_t B_BYTES = KSUB * B_SUB;
constexpr uint32_t SFA_BYTES = KSUB * SFA_SUB;   // the second word only with group-32 scales
constexpr uint32_t SFB_BYTES = KSUB * SFB_SUB;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr uint32_t NUM_BARS = 4 * STAGES + 4;   // full, ready, empty, sf_ready; tmem_full, tmem_empty, done, cp_done
constexpr uint32_t OFF_TMEM_PTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_PTR + 4;
constexpr int kMaxExperts = 1024;
constexpr uint32_t OFF_ENDS = (OFF_ABORT + 4 + 15) / 16 * 16;          // ends[E]
constexpr uint32_t OFF_PFX = OFF_ENDS + kMaxExperts * 4;                // pair tiles before expert e, E + 1
constexpr uint32_t OFF_STG = (OFF_PFX + (kMaxExperts + 1) * 4 + 15) / 16 * 16;
// SiLU window: |g| in [2^-2, 2^6) (exponent field 125..132), 1024 patterns
// of each sign.
constexpr uint32_t kWinB = 125u << 7;
constexpr uint32_t kWinH = 8u * 128u;
constexpr uint32_t OFF_WIN = OFF_STG + 4 * STG_BYTES;
// CTA 0 only: destination of the odd CTA's per-stage signal copies (never read)
constexpr uint32_t OFF_SINK = OFF_WIN + 2 * kWinH * 4;
constexpr uint32_t SMEM_USED = OFF_SINK + SFA_SUB;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
constexpr uint32_t TMEM_COLS = 512;
// stage s: SFA of k-block b at cols 256 + 32 s + 4 b, SFB of k-block b at
// cols 256 + 32 s + 8 + 8 b (two 4-column halves of 128 weight rows)
constexpr uint32_t TMEM_SF_BASE = 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(TMEM_SF_BASE + 32 * STAGES <= TMEM_COLS, "tensor memory budget");
static_assert(KSUB == 1 || KSUB == 2, "stage size");

__host__ __device__ constexpr uint32_t idesc_base(bool b_fp4) {
  return (0u << 7) | ((b_fp4 ? 5u : 0u) << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
         ((uint32_t)(256 >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_even(uint32_t saddr) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(saddr));
  return remote;
}
// Arrive on the barrier at the same shared-memory offset in CTA 0 of the pair
// (epilogue warps releasing the accumulators, after tcgen05.wait::ld).
__device__ __forceinline__ void arrive_even(uint32_t bar, uint32_t rank) {
  if (rank == 0) {
    mbar_arrive(bar);
  } else {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(map_to_even(bar)) : "memory");
  }
}
// The odd CTA's per-stage signal: an asynchronous copy of its transposed
// activation scales (already fenced for the async proxy) into CTA 0's sink,
// completing its bytes on CTA 0's `ready` barrier. The copy reads the very
// words CTA 0's scale-factor copy reads next, through the same proxy, and no
// thread waits on a cross-CTA release.
__device__ __forceinline__ void signal_even_by_copy(uint32_t sink, uint32_t src, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   map_to_even(sink)),
               "r"(src), "r"(SFA_SUB), "r"(map_to_even(bar))
               : "memory");
}
__device__ __forceinline__ void cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Completion of the issuing thread's tcgen05 operations arrives on `bar` in
// this CTA only.
__device__ __forceinline__ void commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Completion of the issuing thread's tcgen05 operations arrives on `bar` in
// both CTAs of the pair.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"((uint16_t)3)
               : "memory");
}

// Bounded wait, as wait_phase, for a barrier that the other CTA of the pair
// also arrives on: the acquire is at cluster scope.
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
static __device__ __noinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                      uint32_t* err) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      *abort_flag = 1;
      raise_error(err, MOE_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Pair tile mp (row tiles counted over the experts): its expert and first row.
__device__ __forceinline__ void pair_tile(const int32_t* ends, const int32_t* pfx, int E, int mp, int& e, int& m0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {  // smallest e with pfx[e + 1] > mp
    const int mid = (lo + hi) >> 1;
    if (pfx[mid + 1] > mp) hi = mid; else lo = mid + 1;
  }
  e = lo;
  const int start = (e == 0) ? 0 : (int)align_up64(ends[e - 1], BM);
  m0 = start + 256 * (mp - pfx[e]);
}
}  // namespace pr

template <bool kBfp4, int kEpi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) grouped_gemm_pair_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const int32_t* __restrict__ a_sf, int ld_sf, const int32_t* __restrict__ ends, int E, int cap,
    const uint32_t* __restrict__ w_sf, int N, int K, uint16_t* __restrict__ out, uint8_t* __restrict__ out_q,
    int32_t* __restrict__ out_sf, int ld_out_sf, float limit, const float* __restrict__ silu_tbl,
    const float* __restrict__ situ_tbl, bool a_g32, bool out_g32, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = pr::cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pr::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pr::OFF_TMEM_PTR);
  const uint32_t bar0 = sbase + pr::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto ready_bar = [&](int s) { return bar0 + 8u * (pr::STAGES + s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * pr::STAGES + s); };
  auto sf_ready_bar = [&](int s) { return bar0 + 8u * (3 * pr::STAGES + s); };
  const uint32_t tmem_full_bar = bar0 + 8u * (4 * pr::STAGES);
  const uint32_t tmem_empty_bar = bar0 + 8u * (4 * pr::STAGES + 1);
  const uint32_t done_bar = bar0 + 8u * (4 * pr::STAGES + 2);
  const uint32_t cp_done_bar = bar0 + 8u * (4 * pr::STAGES + 3);

  // Endpoints and the pair-tile prefix over the experts (warp 0 scans).
  int32_t* ends_s = reinterpret_cast<int32_t*>(smem + pr::OFF_ENDS);
  int32_t* pfx = reinterpret_cast<int32_t*>(smem + pr::OFF_PFX);
  for (int i = threadIdx.x; i < E; i += blockDim.x) ends_s[i] = __ldg(ends + i);
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int start = (e == 0) ? 0 : (int)align_up64(ends_s[e - 1], BM);
        const int c = ends_s[e] - start;
        sum += c > 0 ? (c + 255) / 256 : 0;
      }
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        pfx[e] = run;
        const int start = (e == 0) ? 0 : (int)align_up64(ends_s[e - 1], BM);
        const int c = ends_s[e] - start;
        run += c > 0 ? (c + 255) / 256 : 0;
      }
    }
    if (lane == 31) pfx[E] = incl;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < pr::STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the producer's expect_tx arrive (+ its copies' bytes)
      mbar_init(ready_bar(s), 1);  // CTA 0's transposer (expect_tx) + the odd CTA's signal copy
      mbar_init(empty_bar(s), 1);  // the issuer's multicast commit
      mbar_init(sf_ready_bar(s), 1);  // CTA 0's transposer's commit after the stage's scale copies
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, 8);  // four epilogue warps of each CTA (used in CTA 0)
    mbar_init(done_bar, 1);
    mbar_init(cp_done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(pr::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  pr::cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int KC = K / BK;
  const int KC2 = (KC + pr::KSUB - 1) / pr::KSUB;
  const int n_tiles = N / BN;
  int mpairs = pfx[E];
  const int rows_aligned = (int)align_up64(ends_s[E - 1], BM);
  if (rows_aligned > cap || rows_aligned < 0 || mpairs < 0) {
    if (threadIdx.x == 0 && rank == 0 && pair == 0) raise_error(err, MOE_DEVERR_ENDPOINTS);
    mpairs = 0;
  }
  const int num_tiles = mpairs * n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ producer (each CTA)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
      int s = 0;
      uint32_t ph = 0;
      int issued[pr::STAGES];
      for (int i = 0; i < pr::STAGES; ++i) issued[i] = -1;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
        int e, m0p;
        pr::pair_tile(ends_s, pfx, E, tile / n_tiles, e, m0p);
        const int n0 = (tile % n_tiles) * BN;
        const int m0 = m0p + BM * (int)rank;
        const bool live = m0 < ends_s[e];
        for (int kc2 = 0; kc2 < KC2; ++kc2) {
          const int kc0 = pr::KSUB * kc2, nsub = KC - kc0 < pr::KSUB ? KC - kc0 : pr::KSUB;
          // group-128 scales: the stage's k-blocks sit in one word (KSUB <= 2 and
          // kc0 a multiple of KSUB)
          const int nsfa = a_g32 ? nsub : 1;
          const uint32_t bytes = nsub * ((kBfp4 ? pr::B_SUB / 2 : pr::B_SUB) + pr::SFB_SUB) +
                                 (live ? nsub * pr::A_SUB + nsfa * pr::SFA_SUB : 0u);
          if (!(ok = wait_phase_fast(empty_bar(s), ph ^ 1u, abort_flag, err))) break;
          mbar_arrive_expect_tx(full_bar(s), bytes);
          for (int b = 0; b < nsub; ++b) {
            const int kc = kc0 + b;
            if (live) {
              if (b < nsfa)
                bulk_load(sbase + pr::OFF_SFA + s * pr::SFA_BYTES + b * pr::SFA_SUB,
                          a_sf + (size_t)(a_g32 ? kc : (kc >> 2)) * ld_sf + m0, pr::SFA_SUB, full_bar(s));
              tma_load_2d(sbase + pr::OFF_A + s * pr::A_BYTES + b * pr::A_SUB, &tmA, kc * BK, m0, full_bar(s));
            }
            tma_load_2d(sbase + pr::OFF_B + s * pr::B_BYTES + b * pr::B_SUB, &tmB, kc * BK,
                        e * N + n0 + (BN / 2) * (int)rank, full_bar(s));
            bulk_load(sbase + pr::OFF_SFB + s * pr::SFB_BYTES + b * pr::SFB_SUB, w_sf + ((size_t)e * KC + kc) * N + n0,
                      pr::SFB_SUB, full_bar(s));
          }
          issued[s] = (int)ph;
          if (++s == pr::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // copies already issued complete this CTA's full barriers: let them land
        for (int i = 0; i < pr::STAGES; ++i)
          if (issued[i] >= 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(full_bar(i), (uint32_t)issued[i]) && globaltimer_ns() - t0 < 2000000ull) {}
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (CTA 0)
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      const uint32_t ibase = pr::idesc_base(kBfp4);
      // shared-memory descriptors of stage 0's operands; a stage, a k-block
      // within it and a 32-byte K step move only the start-address field (16-byte units)
      const uint64_t da0 = desc_sw128(sbase + pr::OFF_A), db0 = desc_sw128(sbase + pr::OFF_B);
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
        if (!(ok = pr::wait_phase_cluster(tmem_empty_bar, acc_ph ^ 1u, abort_flag, err))) break;
        tc_fence_after();
        for (int kc2 = 0; kc2 < KC2; ++kc2) {
          // The stage's operands are in shared memory and its scale factors in
          // tensor memory once `sf_ready` completes (the transposer's commit
          // after its scale copies, which it issued once both CTAs' scale
          // words were in place); no further fence is needed for them.
          if (!(ok = wait_phase_fast(sf_ready_bar(s), ph, abort_flag, err))) break;
          const int kc0 = pr::KSUB * kc2, nsub = KC - kc0 < pr::KSUB ? KC - kc0 : pr::KSUB;
          const uint32_t tsf = tmem + pr::TMEM_SF_BASE + 32u * s;
          for (int b = 0; b < nsub; ++b) {
            const int kc = kc0 + b;
            const uint32_t tsfa = tsf + (a_g32 ? 4u * b : 0u), tsfb = tsf + 8u + 8u * b;
            const uint64_t da = da0 + ((s * pr::A_BYTES + b * pr::A_SUB) >> 4);
            const uint64_t db = db0 + ((s * pr::B_BYTES + b * pr::B_SUB) >> 4);
            const uint32_t ib = ibase | ((uint32_t)(kc & 3) << 29);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const uint32_t idesc = a_g32 ? (ibase | ((uint32_t)k4 << 4) | ((uint32_t)k4 << 29)) : (ib | ((uint32_t)k4 << 4));
              pr::mma_pair(tmem, da + 2u * k4, db + 2u * k4, idesc, tsfa, tsfb, (kc | k4) != 0);
            }
          }
          pr::commit_pair(empty_bar(s));
          if (++s == pr::STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        pr::commit_pair(tmem_full_bar);
        acc_ph ^= 1u;
      }
      pr::commit_pair(done_bar);
      wait_phase(done_bar, 0, abort_flag, err, false);
    }
  } else if (warp == 2) {
    // ---------------------------------- activation-scale transposer (each CTA)
    // The copy lands the 128 scale words of the CTA's rows in row order;
    // tcgen05.cp 32x128b.warpx4 wants word (i, j) of its 32 x 4 source at
    // 16 i + 4 j to hold row 32 j + i: lane i reads rows i, 32+i, 64+i, 96+i,
    // then (after the whole warp has read) writes them in place.
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
      int e, m0p;
      pr::pair_tile(ends_s, pfx, E, tile / n_tiles, e, m0p);
      const bool live = m0p + BM * (int)rank < ends_s[e];
      for (int kc2 = 0; kc2 < KC2; ++kc2) {
        const int kc0 = pr::KSUB * kc2, nsub = KC - kc0 < pr::KSUB ? KC - kc0 : pr::KSUB;
        const int nsfa = a_g32 ? nsub : 1;
        if (!(ok = wait_phase_fast(full_bar(s), ph, abort_flag, err))) break;
        if (live) {
          for (int b = 0; b < nsfa; ++b) {
            uint32_t* w = reinterpret_cast<uint32_t*>(smem + pr::OFF_SFA + s * pr::SFA_BYTES + b * pr::SFA_SUB);
            uint4 v;
            v.x = w[lane];
            v.y = w[32 + lane];
            v.z = w[64 + lane];
            v.w = w[96 + lane];
            __syncwarp();
            *reinterpret_cast<uint4*>(w + 4 * lane) = v;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive_expect_tx(ready_bar(s), pr::SFA_SUB);
          else
            pr::signal_even_by_copy(sbase + pr::OFF_SINK, sbase + pr::OFF_SFA + s * pr::SFA_BYTES, ready_bar(s));
        }
        if (++s == pr::STAGES) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp == 3) {
    if (lane == 0 && rank == 0) {
      // -------------------------------------- scale-factor copier (CTA 0)
      // Once both CTAs' scale words of a stage are in place (`ready`), copy
      // them into each CTA's tensor memory (tcgen05.cp.cta_group::2 reads
      // each CTA's own shared memory) and release the issuer by a commit. A
      // thread of its own: a copy takes about as long to issue as an MMA.
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
        for (int kc2 = 0; kc2 < KC2; ++kc2) {
          const int kc0 = pr::KSUB * kc2, nsub = KC - kc0 < pr::KSUB ? KC - kc0 : pr::KSUB;
          if (!(ok = wait_phase_fast(ready_bar(s), ph, abort_flag, err))) break;
          const uint32_t tsf = tmem + pr::TMEM_SF_BASE + 32u * s;
          const uint32_t sfa_s = sbase + pr::OFF_SFA + s * pr::SFA_BYTES;
          const uint32_t sfb_s = sbase + pr::OFF_SFB + s * pr::SFB_BYTES;
          for (int b = 0; b < nsub; ++b) {
            if (b == 0 || a_g32) pr::cp_sf_pair(tsf + 4u * b, desc_sf(sfa_s + b * pr::SFA_SUB));
            pr::cp_sf_pair(tsf + 8u + 8u * b, desc_sf(sfb_s + b * pr::SFB_SUB));
            pr::cp_sf_pair(tsf + 12u + 8u * b, desc_sf(sfb_s + b * pr::SFB_SUB + 512u));
          }
          pr::commit_local(sf_ready_bar(s));
          if (++s == pr::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      // the copies complete before the tensor memory is released
      pr::commit_local(cp_done_bar);
      wait_phase(cp_done_bar, 0, abort_flag, err, false);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue (each CTA)
    const int q = warp & 3;
    const float silu_limit = (kEpi == kEpiSiluClamp) ? spec_silu(limit) : 0.0f;
    float* win = reinterpret_cast<float*>(smem + pr::OFF_WIN);
    if (kEpi == kEpiSilu || kEpi == kEpiSiluClamp) {
      for (int i = threadIdx.x - 128; i < (int)(2 * pr::kWinH); i += 128)
        win[i] = __ldg(silu_tbl + (i < (int)pr::kWinH ? pr::kWinB + i : 0x8000u + pr::kWinB + (i - pr::kWinH)));
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    uint32_t acc_ph = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs) {
      int e, m0p;
      pr::pair_tile(ends_s, pfx, E, tile / n_tiles, e, m0p);
      const int n0 = (tile % n_tiles) * BN;
      const int m0 = m0p + BM * (int)rank;
      const int row_end = ends_s[e];
      if (!wait_phase(tmem_full_bar, acc_ph, abort_flag, err)) break;
      tc_fence_after();
      uint32_t packed[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 32; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + 32u * c, r0);
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + 32u * (c + 1), r1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          packed[16 * c + i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
          packed[16 * (c + 1) + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pr::arrive_even(tmem_empty_bar, rank);
      if (m0 < row_end)  // the odd CTA's rows may all lie past the expert's end
        epilogue_tile<kEpi, pr::kWinB, pr::kWinH>(packed, lane, m0 + 32 * q, row_end, n0, N, out, out_q, out_sf, ld_out_sf,
                                          limit, silu_limit, win, silu_tbl, situ_tbl, out_g32,
                                          sbase + pr::OFF_STG + q * STG_BYTES);
      acc_ph ^= 1u;
    }
  }

  // Both CTAs leave their loops (every wait above is bounded), then free the
  // pair's tensor memory together once the issuer's work has drained. When a
  // role of either CTA gave up, signal copies of the odd CTA may still be in
  // flight to CTA 0: both CTAs wait (bounded) for them before exiting.
  tc_fence_before();
  __syncthreads();
  pr::cluster_sync();
  if (threadIdx.x == 0) {
    uint32_t peer_flag;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(peer_flag)
                 : "r"(sbase + pr::OFF_ABORT), "r"(rank ^ 1u));
    int peer;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer) : "r"(peer_flag) : "memory");
    if (*abort_flag || peer) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {}
    }
  }
  __syncthreads();
  pr::cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(pr::TMEM_COLS) : "memory");
  }
}

template <bool kBfp4, int kEpi>
int launch_impl(const GemmArgs& g, EncodeTiledFn encode, int num_sms, uint32_t* err, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  if (!encode_2d(encode, &tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a, (uint64_t)g.K, (uint64_t)g.cap,
                 (uint64_t)g.K, BK, BM))
    return MOE_ERR_INVALID_ARG;
  const uint64_t wrows = (uint64_t)g.E * (uint64_t)g.N;
  const bool ok = kBfp4 ? encode_2d(encode, &tmB, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w, (uint64_t)g.K,
                                    wrows, (uint64_t)g.K / 2, BK, BN)
                        : encode_2d(encode, &tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w, (uint64_t)g.K, wrows,
                                    (uint64_t)g.K, BK, BN);
  if (!ok) return MOE_ERR_INVALID_ARG;
  const long max_tiles = (long)(g.cap / BM) * (g.N / BN);
  const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  if (grid <= 0) return MOE_OK;
  grouped_gemm_kernel<kBfp4, kEpi><<<grid, kThreads, SMEM_BYTES, st>>>(
      tmA, tmB, g.a_sf, g.ld_sf, g.expert_ends, g.E, g.cap, g.w_sf, g.N, g.K, g.out, g.out_q, g.out_sf,
      g.ld_out_sf, g.limit, g.silu_tbl, g.situ_tbl, (g.w_format & MOE_GEMM_A_GROUP32) != 0, g.out_group == 32, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <bool kBfp4, int kEpi>
int launch_pair_impl(const GemmArgs& g, EncodeTiledFn encode, int max_pairs, uint32_t* err, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  if (!encode_2d(encode, &tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a, (uint64_t)g.K, (uint64_t)g.cap,
                 (uint64_t)g.K, BK, BM))
    return MOE_ERR_INVALID_ARG;
  const uint64_t wrows = (uint64_t)g.E * (uint64_t)g.N;
  const bool ok = kBfp4 ? encode_2d(encode, &tmB, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w, (uint64_t)g.K,
                                    wrows, (uint64_t)g.K / 2, BK, BN / 2)
                        : encode_2d(encode, &tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w, (uint64_t)g.K, wrows,
                                    (uint64_t)g.K, BK, BN / 2);
  if (!ok) return MOE_ERR_INVALID_ARG;
  // pair tiles never outnumber the live 128-row tiles (sizes only, never counts)
  const long max_tiles = (long)(g.cap / BM) * (g.N / BN);
  const int pairs = (int)(max_tiles < max_pairs ? max_tiles : max_pairs);
  if (pairs <= 0) return MOE_OK;
  grouped_gemm_pair_kernel<kBfp4, kEpi><<<2 * pairs, kThreads, pr::SMEM_BYTES, st>>>(
      tmA, tmB, g.a_sf, g.ld_sf, g.expert_ends, g.E, g.cap, g.w_sf, g.N, g.K, g.out, g.out_q, g.out_sf,
      g.ld_out_sf, g.limit, g.silu_tbl, g.situ_tbl, (g.w_format & MOE_GEMM_A_GROUP32) != 0, g.out_group == 32, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The pair kernel computes 256-row tiles: an expert's last tile leaves the odd
// CTA idle when it holds 128 rows or fewer. With few rows per expert (the
// routed rows estimated from the capacity, cap >= routes + E (A - 1), never
// from counts, so that a captured launch stays valid) most pair tiles would
// be half idle, and the one-CTA kernel's 128-row tiles do better.
constexpr long kPairMinRowsPerExpert = 160;

template <int kEpi>
int launch_fmt(const GemmArgs& g, EncodeTiledFn encode, int num_sms, int pairs, bool force_pairs, uint32_t* err,
               cudaStream_t st) {
  const bool fp4 = !(g.w_format & MOE_GEMM_W_E4M3);
  const bool rows_enough = (long)g.cap - 127L * g.E >= kPairMinRowsPerExpert * g.E;
  if (pairs > 0 && g.E <= pr::kMaxExperts && (force_pairs || rows_enough))
    return fp4 ? launch_pair_impl<true, kEpi>(g, encode, pairs, err, st)
               : launch_pair_impl<false, kEpi>(g, encode, pairs, err, st);
  return fp4 ? launch_impl<true, kEpi>(g, encode, num_sms, err, st)
             : launch_impl<false, kEpi>(g, encode, num_sms, err, st);
}

}  // namespace

cudaError_t init_grouped_gemm() {
  const void* fns[] = {
      (const void*)grouped_gemm_kernel<true, kEpiBf16>,  (const void*)grouped_gemm_kernel<false, kEpiBf16>,
      (const void*)grouped_gemm_kernel<true, kEpiSilu>,  (const void*)grouped_gemm_kernel<false, kEpiSilu>,
      (const void*)grouped_gemm_kernel<true, kEpiSiluClamp>, (const void*)grouped_gemm_kernel<false, kEpiSiluClamp>,
      (const void*)grouped_gemm_kernel<true, kEpiSitu>,  (const void*)grouped_gemm_kernel<false, kEpiSitu>};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  const void* pfns[] = {
      (const void*)grouped_gemm_pair_kernel<true, kEpiBf16>,  (const void*)grouped_gemm_pair_kernel<false, kEpiBf16>,
      (const void*)grouped_gemm_pair_kernel<true, kEpiSilu>,  (const void*)grouped_gemm_pair_kernel<false, kEpiSilu>,
      (const void*)grouped_gemm_pair_kernel<true, kEpiSiluClamp>,
      (const void*)grouped_gemm_pair_kernel<false, kEpiSiluClamp>,
      (const void*)grouped_gemm_pair_kernel<true, kEpiSitu>,  (const void*)grouped_gemm_pair_kernel<false, kEpiSitu>};
  for (const void* f : pfns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pr::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// CTA pairs of the pair kernel that fit on the current device at once (one
// pair per two SMs where the hardware can co-schedule them); 0 disables the
// pair kernel.
int grouped_gemm_pairs() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pr::SMEM_BYTES;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)grouped_gemm_pair_kernel<true, kEpiBf16>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int launch_grouped_gemm(const GemmArgs& g, EncodeTiledFn encode, int num_sms, int pairs, bool force_pairs,
                        uint32_t* err, cudaStream_t st) {
  if (g.epi == 1) return launch_fmt<kEpiSilu>(g, encode, num_sms, pairs, force_pairs, err, st);
  if (g.epi == 2) return launch_fmt<kEpiSiluClamp>(g, encode, num_sms, pairs, force_pairs, err, st);
  if (g.epi == 3) return launch_fmt<kEpiSitu>(g, encode, num_sms, pairs, force_pairs, err, st);
  return launch_fmt<kEpiBf16>(g, encode, num_sms, pairs, force_pairs, err, st);
}

}  // namespace moe
