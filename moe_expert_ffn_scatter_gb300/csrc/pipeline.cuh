// pipeline.cuh -- mbarrier and bulk-copy helpers for the streamed kernels:
// a producer thread moves tiles global -> shared with cp.async.bulk and
// counts their bytes on a "full" barrier; consumers release a stage on its
// "empty" barrier. Every wait is bounded by kPipeWaitNs of %globaltimer; a
// wait that runs out raises MOE_DEVERR_WAIT_TIMEOUT and an abort flag in
// shared memory so that the other roles stop waiting too.
#pragma once

#include "common.cuh"

namespace moe {

constexpr unsigned long long kPipeWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void pipe_mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void pipe_mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void pipe_mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool pipe_mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t pipe_globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase of `bar` with parity `parity`. Returns false
// when the wait ran out (error bit and abort flag set) or, with
// honour_abort, when another role has aborted.
static __device__ __noinline__ bool pipe_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t* err,
                                       bool honour_abort = true) {
  if (pipe_mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = pipe_globaltimer();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (pipe_mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if (pipe_globaltimer() - t0 > kPipeWaitNs) {
      *abort_flag = 1;
      raise_error(err, MOE_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Untiled bulk copy global -> shared: both addresses 16-byte aligned, size a
// multiple of 16; completion counted on `bar` in bytes.
__device__ __forceinline__ void pipe_bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Programmatic dependent launch: a kernel launched with the
// programmatic-stream-serialization attribute may start while the previous
// kernel of the stream is still running; pdl_wait() blocks until that kernel
// has completed and its writes are visible (a no-op for a normal launch).
// pdl_launch_dependents() lets the next such kernel start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier over the first `threads` threads of the block (named barrier id).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Arrival on a named barrier without waiting for it (the producer side of a
// producer / consumer hand-over; the consumers bar.sync on the same id).
__device__ __forceinline__ void named_barrier_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Launch, optionally with programmatic stream serialization (the kernel may
// start before the previous kernel of the stream has finished).
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                             Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace moe
