// kernels.h -- internal launchers of the library (host side, not exported).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

inline long lmin(long a, long b) { return a < b ? a : b; }
inline long lmax(long a, long b) { return a > b ? a : b; }

// Tokens per scatter chunk: the unit of the per-chunk expert histogram.
constexpr int kScatterChunk = 64;

size_t route_scatter_ws_bytes(int T, int E, int k);
// Shared memory of a scatter block for rows of H columns (the per-warp stashes)
// and its upper limit: larger H are refused by the route/scatter entry points.
size_t scatter_stash_bytes(int H, bool g32);
constexpr size_t kScatterStashMax = 227 * 1024;
cudaError_t init_route_scatter();
size_t route_scatter_noalloc_max_bytes();
cudaError_t route_scatter_noalloc_scratch(void** addr);
cudaError_t launch_route_scatter_noalloc(const moe_route_args& a, void* scratch, int num_sms, uint32_t* err,
                                         cudaStream_t st);
cudaError_t launch_expert_ends(const int32_t* counts, int E, int A, int32_t* ends, uint32_t* err,
                               cudaStream_t st);
cudaError_t launch_route_scatter(const moe_route_args& a, int num_sms, uint32_t* err, cudaStream_t st);
// 65,536-entry table of spec_silu over all bf16 bit patterns (per context).
cudaError_t launch_silu_table(float* tbl, cudaStream_t st);
// 2 x 65,536 entries: SiTU gate' then up' over all bf16 bit patterns.
cudaError_t launch_situ_table(float* tbl, float beta_s, float beta_l, cudaStream_t st);
cudaError_t launch_act_quant(const uint16_t* gateup, uint8_t* out, int32_t* out_sf,
                             const int32_t* expert_ends, int E, int A, int M_alloc, int I, int kind,
                             float limit, const float* silu_tbl, const float* situ_tbl, int group, int num_sms,
                             uint32_t* err, cudaStream_t st);
cudaError_t launch_combine(const uint16_t* down, int H, const float* topk_w, const int32_t* src2dst,
                           int T, int k, float rsf, uint16_t* out, int num_sms, cudaStream_t st);
cudaError_t launch_prepare_weights(const uint8_t* w_in, const uint8_t* sf_in, int E, int N, int K,
                                   int w_format, uint8_t* w_out, uint32_t* sf_out, cudaStream_t st);

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct GemmArgs {
  const uint8_t* a;
  const int32_t* a_sf;
  int ld_sf;
  const int32_t* expert_ends;
  int E, cap;
  const uint8_t* w;
  const uint32_t* w_sf;
  int w_format;
  int N, K;
  uint16_t* out;
  // Fused GEMM1 epilogue (epi 1: SiLU*mul, 2: with clamp `limit`): the
  // weights' gate/up rows are interleaved in blocks of 128 and the kernel
  // writes e4m3 codes [cap, N/2] and packed scales [N/512][ld_out_sf]
  // instead of `out`.
  int epi = 0;
  uint8_t* out_q = nullptr;
  int32_t* out_sf = nullptr;
  int ld_out_sf = 0;
  float limit = 0.0f;
  const float* silu_tbl = nullptr;
  const float* situ_tbl = nullptr;
  int out_group = 128;  // group of the fused epilogue's e4m3 output: 128, or 32
};
// Per-device set-up (shared-memory opt-in); called once per context.
cudaError_t init_grouped_gemm();
// CTA pairs of the pair kernel resident at once on the current device (0: the
// one-CTA kernel only); queried once per context.
int grouped_gemm_pairs();
// Returns MOE_OK or a MOE_ERR_* code. The CTA-pair kernel (at most `pairs`
// pairs) runs when pairs > 0, E <= 1024 and either `force_pairs` or the
// capacity holds at least 160 routed rows per expert beyond the alignment
// gaps (cap - 127 E >= 160 E); otherwise the one-CTA kernel.
int launch_grouped_gemm(const GemmArgs& g, EncodeTiledFn encode, int num_sms, int pairs, bool force_pairs,
                        uint32_t* err, cudaStream_t st);

cudaError_t init_decode();
// mma.sync path when allowed and applicable (decode_mma_sync_ok), else the
// per-(token, slot) GEMV launches.
bool decode_mma_sync_ok(const moe_decode_args& a);
cudaError_t launch_decode(const moe_decode_args& a, bool allow_mma_sync, int num_sms, uint32_t* err,
                          cudaStream_t st);
// out = slot-ordered weighted sum of y2 over local slots (last launch of both
// decode paths); pdl: may start before the previous kernel has finished.
cudaError_t launch_weighted_sum(const moe_decode_args& a, bool pdl, cudaStream_t st);

// Workspace of the tcgen05 decode path: byte offsets of its regions (each
// 1024-byte aligned) and the segment-row capacity R.
struct DecodeWs {
  size_t cnt, seg, row_slot, xs, xsf, as, asf, total;
  int R;
};
DecodeWs decode_ws_layout(int T, int k, int H, int I, int n_local);
bool decode_gemm_ok(int T, int k, int H, int I, int n_local, int wfmt);
cudaError_t init_decode_gemm();
// Returns MOE_OK or a MOE_ERR_* code; a.workspace holds decode_ws_layout().total bytes.
int launch_decode_gemm(const moe_decode_args& a, EncodeTiledFn enc, int num_sms, uint32_t* err, cudaStream_t st);

}  // namespace moe
