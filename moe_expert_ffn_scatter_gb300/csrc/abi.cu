// abi.cu -- the exported C entry points: context, argument validation and
// the launch sequence of each call. See include/moe_gb300.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <stdlib.h>

#include "moe_gb300.h"
#include "kernels.h"

struct moe_ctx {
  int device;
  int num_sms;
  int gemm_pairs;         // CTA pairs of the pair GEMM kernel resident at once (0: one-CTA kernel)
  bool gemm_pairs_forced;  // take the pair kernel whatever the rows per expert
  uint32_t* d_err;
  float* d_silu;  // 65,536-entry SiLU table of the exp/SiLU specification
  float* d_situ;  // 2 x 65,536-entry SiTU tables (gate', up') for situ_bs / situ_bl
  float situ_bs, situ_bl;
  void* d_route_scratch;  // device address of the built-in scratch of moe_route_scatter_noalloc
  moe::EncodeTiledFn encode;
};

namespace {

inline cudaStream_t S(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline long align4l(long n) { return (n + 3) / 4 * 4; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Every call runs on the context's device.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

MOE_API int moe_version(void) { return 10000; }

MOE_API const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CAPACITY: return "capacity below the routed rows plus alignment gaps";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or device";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE: return "device-side error";
    default: return "unknown status";
  }
}

MOE_API int moe_ctx_create(moe_ctx** out, int device) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_CUDA;
  DeviceGuard g(device);
  if (!g.ok) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  moe_ctx* c = static_cast<moe_ctx*>(calloc(1, sizeof(moe_ctx)));
  if (!c) return MOE_ERR_CUDA;
  c->device = device;
  c->num_sms = prop.multiProcessorCount;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    free(c);
    return MOE_ERR_CUDA;
  }
  c->encode = reinterpret_cast<moe::EncodeTiledFn>(fn);
  if (cudaMalloc(&c->d_err, sizeof(uint32_t)) != cudaSuccess) {
    free(c);
    return MOE_ERR_CUDA;
  }
  if (cudaMalloc(&c->d_silu, 65536 * sizeof(float)) != cudaSuccess) {
    cudaFree(c->d_err);
    free(c);
    return MOE_ERR_CUDA;
  }
  if (cudaMalloc(&c->d_situ, 2 * 65536 * sizeof(float)) != cudaSuccess) {
    cudaFree(c->d_silu);
    cudaFree(c->d_err);
    free(c);
    return MOE_ERR_CUDA;
  }
  c->situ_bs = 4.0f;  // Kimi's SiTU pair, filled now so that ordinary use never refills
  c->situ_bl = 25.0f;
  if (moe::init_grouped_gemm() != cudaSuccess || moe::init_route_scatter() != cudaSuccess ||
      moe::init_decode() != cudaSuccess ||
      moe::init_decode_gemm() != cudaSuccess ||
      cudaMemset(c->d_err, 0, sizeof(uint32_t)) != cudaSuccess ||
      moe::launch_silu_table(c->d_silu, 0) != cudaSuccess ||
      moe::launch_situ_table(c->d_situ, c->situ_bs, c->situ_bl, 0) != cudaSuccess ||
      moe::route_scatter_noalloc_scratch(&c->d_route_scratch) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(c->d_situ);
    cudaFree(c->d_silu);
    cudaFree(c->d_err);
    free(c);
    return MOE_ERR_CUDA;
  }
  c->gemm_pairs = moe::grouped_gemm_pairs();  // after the shared-memory opt-in above
  if (const char* cap_pairs = getenv("MOE_GEMM_CTA_PAIRS")) {
    const long v = strtol(cap_pairs, nullptr, 10);
    if (v >= 0 && v < c->gemm_pairs) c->gemm_pairs = (int)v;
    c->gemm_pairs_forced = v > 0;
  }
  *out = c;
  return MOE_OK;
}

MOE_API int moe_ctx_destroy(moe_ctx* ctx) {
  if (!ctx) return MOE_OK;
  DeviceGuard g(ctx->device);
  cudaFree(ctx->d_silu);
  cudaFree(ctx->d_situ);
  cudaFree(ctx->d_err);
  free(ctx);
  return MOE_OK;
}

MOE_API int moe_get_device_error(moe_ctx* ctx, uint32_t* bits, moe_stream_t stream) {
  if (!ctx || !bits) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, ctx->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, S(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d_err, 0, sizeof(uint32_t), S(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
  *bits = h;
  return cuda_status(e);
}

MOE_API int moe_expert_ends_from_counts(moe_ctx* ctx, const int32_t* counts, int E, int A,
                                        int32_t* expert_ends, moe_stream_t stream) {
  if (!ctx || !counts || !expert_ends || E < 1 || E > 8192 || A < 1) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  return cuda_status(moe::launch_expert_ends(counts, E, A, expert_ends, ctx->d_err, S(stream)));
}

MOE_API size_t moe_route_scatter_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return moe::route_scatter_ws_bytes(T, E, k);
}

// Argument checks shared by moe_route_scatter and moe_route_scatter_noalloc
// (everything but the scratch: the caller's workspace, or the built-in array).
static int check_route_args(const moe_route_args* a) {
  if (a->T < 0 || a->E < 1 || a->E > 4096 || a->k < 1 || a->k > 32 || a->k > a->E || a->H < 128 ||
      a->H % 128 != 0 || a->A < 1 || a->cap < 0 ||
      (a->quant_group != 0 && a->quant_group != 128 && a->quant_group != 32))
    return MOE_ERR_INVALID_ARG;
  if (a->routing_mode != MOE_ROUTE_SOFTMAX_TOPK && a->routing_mode != MOE_ROUTE_SIGMOID_BIAS_TOPK &&
      a->routing_mode != MOE_ROUTE_PRECOMPUTED)
    return MOE_ERR_INVALID_ARG;
  if (a->routing_mode != MOE_ROUTE_PRECOMPUTED && (a->E > 1024 || !a->logits || !a->topk_w))
    return MOE_ERR_INVALID_ARG;
  if (a->routing_mode == MOE_ROUTE_SIGMOID_BIAS_TOPK && !a->corr_bias) return MOE_ERR_INVALID_ARG;
  if (!a->expert_ends) return MOE_ERR_INVALID_ARG;
  if (a->T > 0 && (!a->topk_ids || !a->x || !a->a_fp8 || !a->a_sf || !a->src2dst)) return MOE_ERR_INVALID_ARG;
  if (a->T > 0 && (!al(a->x, 16) || !al(a->a_fp8, 8) || !al(a->a_sf, 4))) return MOE_ERR_INVALID_ARG;
  if ((long)a->cap < (long)a->T * a->k + (long)a->E * (a->A - 1)) return MOE_ERR_CAPACITY;
  if ((long)a->cap * a->H > 0x7FFFFFFFFFFFL) return MOE_ERR_INVALID_ARG;
  if (moe::scatter_stash_bytes(a->H, a->quant_group == 32) > moe::kScatterStashMax) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

MOE_API int moe_route_scatter(moe_ctx* ctx, const moe_route_args* a, moe_stream_t stream) {
  if (!ctx || !a) return MOE_ERR_INVALID_ARG;
  const int rc = check_route_args(a);
  if (rc != MOE_OK) return rc;
  if (!a->workspace || a->workspace_bytes < moe::route_scatter_ws_bytes(a->T, a->E, a->k) || !al(a->workspace, 16))
    return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MOE_ERR_CUDA;
  return cuda_status(moe::launch_route_scatter(*a, ctx->num_sms, ctx->d_err, S(stream)));
}

MOE_API int moe_route_scatter_noalloc(moe_ctx* ctx, const moe_route_args* a, moe_stream_t stream) {
  if (!ctx || !a) return MOE_ERR_INVALID_ARG;
  const int rc = check_route_args(a);
  if (rc != MOE_OK) return rc;
  if (moe::route_scatter_ws_bytes(a->T, a->E, a->k) > moe::route_scatter_noalloc_max_bytes())
    return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MOE_ERR_CUDA;
  return cuda_status(moe::launch_route_scatter_noalloc(*a, ctx->d_route_scratch, ctx->num_sms, ctx->d_err,
                                                       S(stream)));
}

MOE_API int moe_prepare_weights(moe_ctx* ctx, const uint8_t* w_in, const uint8_t* sf_in, int E, int N,
                                int K, int w_format, uint8_t* w_out, uint32_t* sf_out, moe_stream_t stream) {
  if (!ctx || !w_in || !sf_in || !w_out || !sf_out || E < 1 || N < 128 || N % 128 != 0 || K < 128 ||
      K % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if ((w_format & ~(MOE_GEMM_W_E4M3 | MOE_GEMM_W_GATEUP_BLOCK128 | MOE_GEMM_W_IN_E4M3 | MOE_GEMM_W_SF_BLOCK128)) != 0)
    return MOE_ERR_INVALID_ARG;
  if ((w_format & MOE_GEMM_W_IN_E4M3) && !(w_format & MOE_GEMM_W_E4M3)) return MOE_ERR_INVALID_ARG;
  if ((w_format & MOE_GEMM_W_GATEUP_BLOCK128) && N % 256 != 0) return MOE_ERR_INVALID_ARG;
  const bool widen = (w_format & MOE_GEMM_W_E4M3) && !(w_format & MOE_GEMM_W_IN_E4M3);
  if ((widen || (w_format & MOE_GEMM_W_GATEUP_BLOCK128)) && w_out == w_in) return MOE_ERR_INVALID_ARG;
  if (!al(sf_out, 4) || ((w_format & MOE_GEMM_W_E4M3) && !al(w_out, 2))) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  return cuda_status(moe::launch_prepare_weights(w_in, sf_in, E, N, K, w_format, w_out, sf_out, S(stream)));
}

static int check_gemm(const moe::GemmArgs& g) {
  if (!g.a || !g.a_sf || !g.expert_ends || !g.w || !g.w_sf || (g.epi == 0 && !g.out)) return MOE_ERR_INVALID_ARG;
  if (g.E < 1 || g.E > 4096 || g.N < 256 || g.N % 256 != 0 || g.K < 128 || g.K % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (g.cap < 0 || g.cap % 128 != 0 || g.ld_sf < g.cap || g.ld_sf % 4 != 0) return MOE_ERR_INVALID_ARG;
  if ((g.w_format & ~(MOE_GEMM_W_E4M3 | MOE_GEMM_W_GATEUP_BLOCK128 | MOE_GEMM_A_GROUP32)) != 0)
    return MOE_ERR_INVALID_ARG;
  if (!al(g.a, 16) || !al(g.w, 32) || !al(g.a_sf, 16) || !al(g.w_sf, 16)) return MOE_ERR_INVALID_ARG;
  if (g.epi == 0 ? (!al(g.out, 16)) : (!g.out_q || !g.out_sf || !al(g.out_q, 16) || g.N % 256 != 0))
    return MOE_ERR_INVALID_ARG;
  if ((long)g.E * g.N >= (1L << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

MOE_API int moe_grouped_gemm(moe_ctx* ctx, const uint8_t* a, const int32_t* a_sf, int ld_sf,
                             const int32_t* expert_ends, int E, int A, int cap, const uint8_t* w,
                             const uint32_t* w_sf, int w_format, int N, int K, uint16_t* out,
                             moe_stream_t stream) {
  if (!ctx || A != 128) return MOE_ERR_INVALID_ARG;
  moe::GemmArgs g{a, a_sf, ld_sf, expert_ends, E, cap, w, w_sf, w_format, N, K, out};
  int rc = check_gemm(g);
  if (rc != MOE_OK) return rc;
  if (cap == 0) return MOE_OK;
  DeviceGuard dg(ctx->device);
  return moe::launch_grouped_gemm(g, ctx->encode, ctx->num_sms, ctx->gemm_pairs, ctx->gemm_pairs_forced, ctx->d_err, S(stream));
}

// Activation parameters: SiLU, SiLU with a clamp limit L > 0, or SiTU with
// finite positive betas.
static int act_group(const moe_act_params* act) { return act->quant_group == 32 ? 32 : 128; }

static int check_act(const moe_act_params* act) {
  if (act->quant_group != 0 && act->quant_group != 128 && act->quant_group != 32) return MOE_ERR_INVALID_ARG;
  if (act->kind == MOE_ACT_SILU) return MOE_OK;
  if (act->kind == MOE_ACT_SILU_CLAMP) return (act->limit > 0.0f) ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (act->kind == MOE_ACT_SITU)
    return (act->situ_beta_s > 0.0f && act->situ_beta_s < INFINITY && act->situ_beta_l > 0.0f &&
            act->situ_beta_l < INFINITY)
               ? MOE_OK
               : MOE_ERR_INVALID_ARG;
  return MOE_ERR_INVALID_ARG;
}

// SiTU tables for the requested betas, refilled on the call's stream when
// they differ from the ones the context holds.
static int prepare_act(moe_ctx* ctx, const moe_act_params* act, cudaStream_t st) {
  if (act->kind != MOE_ACT_SITU) return MOE_OK;
  if (act->situ_beta_s == ctx->situ_bs && act->situ_beta_l == ctx->situ_bl) return MOE_OK;
  if (moe::launch_situ_table(ctx->d_situ, act->situ_beta_s, act->situ_beta_l, st) != cudaSuccess) return MOE_ERR_CUDA;
  ctx->situ_bs = act->situ_beta_s;
  ctx->situ_bl = act->situ_beta_l;
  return MOE_OK;
}

static int epi_of(const moe_act_params* act) {
  return act->kind == MOE_ACT_SITU ? 3 : (act->kind == MOE_ACT_SILU_CLAMP ? 2 : 1);
}

MOE_API int moe_grouped_gemm_act_quant(moe_ctx* ctx, const uint8_t* a, const int32_t* a_sf, int ld_sf,
                                       const int32_t* expert_ends, int E, int A, int cap, const uint8_t* w13,
                                       const uint32_t* w13_sf, int w_format, int I, int K,
                                       const moe_act_params* act, uint8_t* out_fp8, int32_t* out_sf,
                                       moe_stream_t stream) {
  if (!ctx || !act || A != 128 || !(w_format & MOE_GEMM_W_GATEUP_BLOCK128)) return MOE_ERR_INVALID_ARG;
  if (check_act(act) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (I < 128 || I % 128 != 0) return MOE_ERR_INVALID_ARG;
  moe::GemmArgs g{a, a_sf, ld_sf, expert_ends, E, cap, w13, w13_sf,
                  w_format & (MOE_GEMM_W_E4M3 | MOE_GEMM_A_GROUP32), 2 * I, K, nullptr};
  g.epi = epi_of(act);
  g.out_group = act_group(act);
  g.silu_tbl = ctx->d_silu;
  g.situ_tbl = ctx->d_situ;
  g.out_q = out_fp8;
  g.out_sf = out_sf;
  g.ld_out_sf = (int)align4l(cap);
  g.limit = act->limit;
  int rc = check_gemm(g);
  if (rc != MOE_OK) return rc;
  if (!al(out_sf, 4)) return MOE_ERR_INVALID_ARG;
  if (cap == 0) return MOE_OK;
  DeviceGuard dg(ctx->device);
  if ((rc = prepare_act(ctx, act, S(stream))) != MOE_OK) return rc;
  return moe::launch_grouped_gemm(g, ctx->encode, ctx->num_sms, ctx->gemm_pairs, ctx->gemm_pairs_forced, ctx->d_err, S(stream));
}

MOE_API int moe_act_quant(moe_ctx* ctx, const uint16_t* gateup, uint8_t* out, int32_t* out_sf,
                          const int32_t* expert_ends, int E, int A, int M_alloc, int I,
                          const moe_act_params* act, moe_stream_t stream) {
  if (!ctx || !act || M_alloc < 0 || I < 128 || I % 128 != 0 || A < 1) return MOE_ERR_INVALID_ARG;
  if (M_alloc > 0 && (!gateup || !out || !out_sf)) return MOE_ERR_INVALID_ARG;
  if (expert_ends && (E < 1 || E > 65535)) return MOE_ERR_INVALID_ARG;
  if (check_act(act) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (!al(gateup, 16) || !al(out, 16) || !al(out_sf, 4)) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  const int rc = prepare_act(ctx, act, S(stream));
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_act_quant(gateup, out, out_sf, expert_ends, E, A, M_alloc, I, act->kind,
                                           act->limit, ctx->d_silu, ctx->d_situ, act_group(act), ctx->num_sms,
                                           ctx->d_err, S(stream)));
}

MOE_API int moe_combine(moe_ctx* ctx, const uint16_t* down, int H, const float* topk_w,
                        const int32_t* src2dst, int T, int k, float rsf, uint16_t* out, moe_stream_t stream) {
  if (!ctx || T < 0 || k < 1 || H < 8 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!down || !topk_w || !src2dst || !out)) return MOE_ERR_INVALID_ARG;
  if (!al(down, 16) || !al(out, 16)) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  return cuda_status(moe::launch_combine(down, H, topk_w, src2dst, T, k, rsf, out, ctx->num_sms, S(stream)));
}

MOE_API int moe_ffn_forward(moe_ctx* ctx, const moe_ffn_args* a, moe_stream_t stream) {
  if (!ctx || !a) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->k < 1 || a->A != 128 || a->H % 256 != 0 || a->I % 128 != 0 || (2 * a->I) % 256 != 0 ||
      a->cap % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  const bool fused = (a->w_format & MOE_GEMM_W_GATEUP_BLOCK128) != 0;
  if ((!fused && !a->gateup) || !a->act_fp8 || !a->act_sf || !a->down || !a->topk_w || !a->src2dst || !a->out)
    return MOE_ERR_INVALID_ARG;
  if (check_act(&a->act) != MOE_OK) return MOE_ERR_INVALID_ARG;
  const int ld = (int)align4l(a->cap);
  const int fmt = a->w_format & MOE_GEMM_W_E4M3;
  // GEMM1 reads the scatter's scales (their group: the A_GROUP32 flag of
  // w_format); GEMM2 reads the act-quant's (their group: act.quant_group)
  const int fmt2 = fmt | (act_group(&a->act) == 32 ? MOE_GEMM_A_GROUP32 : 0);
  moe::GemmArgs g1{a->a_fp8, a->a_sf, ld, a->expert_ends, a->E, a->cap, a->w13, a->w13_sf,
                   fmt | (a->w_format & MOE_GEMM_A_GROUP32), 2 * a->I, a->H, a->gateup};
  if (fused) {
    g1.silu_tbl = ctx->d_silu;
    g1.situ_tbl = ctx->d_situ;
    g1.epi = epi_of(&a->act);
    g1.out_group = act_group(&a->act);
    g1.out_q = a->act_fp8;
    g1.out_sf = a->act_sf;
    g1.ld_out_sf = ld;
    g1.limit = a->act.limit;
  }
  moe::GemmArgs g2{a->act_fp8, a->act_sf, ld, a->expert_ends, a->E, a->cap, a->w2, a->w2_sf, fmt2,
                   a->H, a->I, a->down};
  int rc;
  if ((rc = check_gemm(g1)) != MOE_OK || (rc = check_gemm(g2)) != MOE_OK) return rc;
  if ((!fused && !al(a->gateup, 16)) || !al(a->act_fp8, 16) || !al(a->act_sf, 4) || !al(a->down, 16) ||
      !al(a->out, 16))
    return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(ctx->device);
  if ((rc = prepare_act(ctx, &a->act, S(stream))) != MOE_OK) return rc;
  if (a->cap > 0) {
    if ((rc = moe::launch_grouped_gemm(g1, ctx->encode, ctx->num_sms, ctx->gemm_pairs, ctx->gemm_pairs_forced, ctx->d_err, S(stream))) != MOE_OK) return rc;
    if (!fused &&
        (rc = cuda_status(moe::launch_act_quant(a->gateup, a->act_fp8, a->act_sf, a->expert_ends, a->E, a->A,
                                                a->cap, a->I, a->act.kind, a->act.limit, ctx->d_silu,
                                                ctx->d_situ, act_group(&a->act), ctx->num_sms, ctx->d_err,
                                                S(stream)))) != MOE_OK)
      return rc;
    if ((rc = moe::launch_grouped_gemm(g2, ctx->encode, ctx->num_sms, ctx->gemm_pairs, ctx->gemm_pairs_forced, ctx->d_err, S(stream))) != MOE_OK) return rc;
  }
  return cuda_status(moe::launch_combine(a->down, a->H, a->topk_w, a->src2dst, a->T, a->k, a->rsf, a->out,
                                         ctx->num_sms, S(stream)));
}

MOE_API size_t moe_decode_workspace_size(int32_t T, int32_t k, int32_t H, int32_t I, int32_t num_local_experts) {
  if (T < 1 || k < 1 || k > 32 || H < 32 || I < 32 || num_local_experts < 1) return 0;
  return moe::decode_ws_layout(T, k, H, I, num_local_experts).total;
}

MOE_API int moe_sparse_gemv_decode(moe_ctx* ctx, const moe_decode_args* a, moe_stream_t stream) {
  if (!ctx || !a) return MOE_ERR_INVALID_ARG;
  const bool ws = a->workspace != nullptr;
  if (a->T < 0 || a->T > (ws ? 128 : 64) || a->k < 1 || a->k > 32 || a->H < 32 || a->H % 32 != 0 || a->I < 32 ||
      a->I % 32 != 0 || a->num_local_experts < 0)
    return MOE_ERR_INVALID_ARG;
  if (a->wfmt != MOE_WFMT_FP8_PER_EXPERT && a->wfmt != MOE_WFMT_MXFP4_G32) return MOE_ERR_INVALID_ARG;
  if (a->glu_layout != MOE_GLU_HALVES && a->glu_layout != MOE_GLU_INTERLEAVED) return MOE_ERR_INVALID_ARG;
  if (a->T > 0) {
    if (!a->x || !a->topk_ids || !a->topk_w || !a->w_gu || !a->b_gu || !a->w_d || !a->b_d || !a->y1 ||
        !a->act || !a->y2 || !a->out)
      return MOE_ERR_INVALID_ARG;
    if (a->wfmt == MOE_WFMT_FP8_PER_EXPERT && (!a->w_gu_scale || !a->w_d_scale)) return MOE_ERR_INVALID_ARG;
    if (a->wfmt == MOE_WFMT_MXFP4_G32 && (!a->w_gu_sf || !a->w_d_sf || !al(a->w_gu_sf, 16) || !al(a->w_d_sf, 16)))
      return MOE_ERR_INVALID_ARG;
    if (!al(a->w_gu, 16) || !al(a->w_d, 16) || !al(a->b_gu, 16) || !al(a->b_d, 16) || !al(a->x, 8) ||
        !al(a->act, 8))
      return MOE_ERR_INVALID_ARG;
  }
  if (a->path < MOE_DECODE_AUTO || a->path > MOE_DECODE_GEMV) return MOE_ERR_INVALID_ARG;
  if (ws && !al(a->workspace, 256)) return MOE_ERR_INVALID_ARG;
  // tcgen05 path: sizes in range, e2m1 tensor maps want a 32-byte aligned base,
  // 16-byte vector stores of y1 / act / y2, and a large enough workspace
  const bool tc5 = ws && a->T > 0 &&
                   moe::decode_gemm_ok(a->T, a->k, a->H, a->I, a->num_local_experts, a->wfmt) &&
                   (a->wfmt != MOE_WFMT_MXFP4_G32 || (al(a->w_gu, 32) && al(a->w_d, 32))) && al(a->y1, 16) &&
                   al(a->act, 16) && al(a->y2, 16) &&
                   a->workspace_bytes >= moe::decode_ws_layout(a->T, a->k, a->H, a->I, a->num_local_experts).total;
  const bool mma = a->T > 0 && moe::decode_mma_sync_ok(*a);
  int path = a->path;
  if (path == MOE_DECODE_AUTO) {
    const int t_min = a->wfmt == MOE_WFMT_FP8_PER_EXPERT ? 8 : 4;  // measured crossover with the mma.sync path
    path = (tc5 && (a->T >= t_min || !mma)) ? MOE_DECODE_TCGEN05 : mma ? MOE_DECODE_MMA_SYNC : MOE_DECODE_GEMV;
  }
  if (a->T > 0 && ((path == MOE_DECODE_TCGEN05 && !tc5) || (path == MOE_DECODE_MMA_SYNC && !mma) ||
                   (path == MOE_DECODE_GEMV && a->T > 64)))
    return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (path == MOE_DECODE_TCGEN05 && a->T > 0)
    return moe::launch_decode_gemm(*a, ctx->encode, ctx->num_sms, ctx->d_err, S(stream));
  return cuda_status(moe::launch_decode(*a, path == MOE_DECODE_MMA_SYNC, ctx->num_sms, ctx->d_err, S(stream)));
}

}  // extern "C"
