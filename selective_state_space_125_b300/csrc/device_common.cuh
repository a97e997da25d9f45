// Device-side helpers shared by the scan and decode kernels: math in fast
// (hardware approximation) and precise (libdevice) forms, bf16/fp32 element
// access, mbarrier + TMA wrappers with bounded waits, and the status word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mamba {

// Kernels never trap: a bounded wait that runs out records kStatusTimeout in
// the device status word (whose address every launch receives) and the kernel
// returns early.
constexpr int kStatusTimeout = 4;

// Default upper bound of every spin-wait in the kernels, in nanoseconds of
// %globaltimer (2 s; a healthy wait is microseconds). The scan and decode
// launches carry the limit of their first waits in their arguments, so that a
// test can shorten it; the waits that drain copies in flight after a timeout
// always use this default.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// |A| floor of the kernels. exp(dt A) and (exp(dt A) - 1) / A at |A| = 1e-20
// equal their A -> 0 limits (1 and dt) in fp32 for any dt below 1e12, and
// 1e-20 keeps A h, dt A and 1 / A inside the normal fp32 range.
constexpr float kMinAbsA = 1e-20f;

// Smallest |dt A| (natural units) at which the bf16 path forms exp(dt A) - 1
// as ex2(dt A log2 e) - 1. The MUFU result carries an absolute error near
// 2^-23, so the relative error of the difference is below 2^-9 there; steps
// with a smaller |dt A| in any lane of the warp take expm1_acc instead.
constexpr float kFastMinDtA = 6.103515625e-05f;  // 2^-14

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void record_status(int* word, int code) {
  if (word) atomicCAS(word, 0, code);
}

// Programmatic dependent launch (sm_90 and later). A kernel launched with the
// programmatic-stream-serialization attribute may start while the kernel
// before it in the stream is still running; griddep_wait() blocks the calling
// thread until that kernel has completed and its memory is visible, so every
// thread calls it before its first global-memory access. griddep_launch()
// lets the next such kernel in the stream start early (it still waits).
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic
// stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- math
// Hardware approximations (MUFU): 2^x, log2(x), 1/x with flush-to-zero.
__device__ __forceinline__ float hw_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float hw_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float hw_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = max(x, 0) + log(1 + e) with e = e^-|x|. Fast form: log(1 + e)
// by lg2 for e >= 2^-10 (relative error about 2^-24 / e <= 2^-14), and by
// e - e^2 / 2 below that (relative error below e^2 / 3 <= 2^-21).
__device__ __forceinline__ float softplus_fast(float x) {
  const float e = hw_ex2(-fabsf(x) * kLog2e);
  const float series = fmaf(-0.5f * e, e, e);
  const float lp = (e < 0.0009765625f) ? series : hw_lg2(1.0f + e) * kLn2;
  return fmaxf(x, 0.0f) + lp;
}
__device__ __forceinline__ float softplus_precise(float x) {
  return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

// exp(x) - 1 for x <= 0 with full relative accuracy, given xl = x log2(e)
// and e = ex2(xl) (a MUFU value): the series x (1 + x/2 + x^2/6 + x^3/24)
// below |x| = 1/8 (truncation error below x^4 / 120 < 2e-6 relative), e - 1
// above it (cancellation error below 2^-23 / (1/8) = 1e-6 relative).
__device__ __forceinline__ float expm1_acc(float xl, float e) {
  const float x = xl * kLn2;
  const float s = x * fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
  return (fabsf(x) < 0.125f) ? s : e - 1.0f;
}

// SiLU(z) = z * sigmoid(z).
__device__ __forceinline__ float silu_fast(float z) { return z * hw_rcp(1.0f + hw_ex2(-z * kLog2e)); }
__device__ __forceinline__ float silu_precise(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------ element access
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// --------------------------------------------------- mbarrier and TMA
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false once limit_ns
// has passed. A limit of 0 gives up at once without polling (a test setting).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 3-D tiled TMA load (tensor map coordinates innermost first) into shared
// memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace mamba
