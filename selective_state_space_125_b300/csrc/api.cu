// C ABI of libmamba_ssm_b300.so (declared in include/mamba_ssm.h): argument
// validation, work planning, TMA descriptor encoding and kernel dispatch.
// Every step of the computation runs in the kernels of scan_kernel.cuh and
// state_update.cu; this file only checks, plans and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "mamba_ssm.h"
#include "bwd_args.h"
#include "decode_args.h"
#include "scan_args.h"

namespace mamba {
cudaError_t launch_scan_f32_d0(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
cudaError_t launch_scan_f32_d1(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
cudaError_t launch_scan_bf16_d0(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
cudaError_t launch_scan_bf16_d1(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
cudaError_t launch_scan_f32_conv(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
cudaError_t launch_scan_bf16_conv(int, int, ScanMode, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
bool scan_variant_f32(int, int, ScanVariant*);
bool scan_variant_bf16(int, int, ScanVariant*);
cudaError_t launch_scan_tp(int, int, const ScanArgs&, const ScanMaps&, dim3, cudaStream_t);
}  // namespace mamba

using namespace mamba;

// Kernel status word, one instance per device (see mamba_device_status).
__device__ int g_mamba_status_word;

namespace {

constexpr int kVersion = 1 * 10000 + 1 * 100 + 0;
constexpr unsigned long long kWaitLimitNsDefault = 2000000000ull;  // the kernels' default wait limit (2 s)
constexpr int kMaxState = 256;
constexpr int kMaxDevices = 64;

thread_local std::string t_detail;

mamba_status_t fail(mamba_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_detail = buf;
  return s;
}

mamba_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MAMBA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, read once with the device current.
mamba_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MAMBA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_mamba_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    di.ready = true;
  }
  *out = di;
  return MAMBA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a row-major (outer, mid, inner) tensor with box (box_inner, box_mid, 1).
mamba_status_t encode_3d(CUtensorMap* map, const void* base, int es, uint64_t inner, uint64_t mid, uint64_t outer,
                         uint32_t box_inner, uint32_t box_mid) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * es, inner * mid * es};
  const cuuint32_t box[3] = {box_inner, box_mid, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = (es == 2) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult %d", int(r));
  return MAMBA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool variant_for(int dtype, int npl, int lpc, ScanVariant* v) {
  return dtype == 0 ? scan_variant_f32(npl, lpc, v) : scan_variant_bf16(npl, lpc, v);
}

// One scan pass for (input dtype, discretisation); the fused-conv kernels
// (zero-order hold only) when the arguments carry conv taps.
cudaError_t launch_scan_pass(int dtype, int disc, int npl, int lpc, ScanMode mode, const ScanArgs& a,
                             const ScanMaps& maps, dim3 grid, cudaStream_t stream) {
  if (a.conv_w)
    return dtype == 0 ? launch_scan_f32_conv(npl, lpc, mode, a, maps, grid, stream)
                      : launch_scan_bf16_conv(npl, lpc, mode, a, maps, grid, stream);
  if (dtype == 0)
    return disc == 0 ? launch_scan_f32_d0(npl, lpc, mode, a, maps, grid, stream)
                     : launch_scan_f32_d1(npl, lpc, mode, a, maps, grid, stream);
  return disc == 0 ? launch_scan_bf16_d0(npl, lpc, mode, a, maps, grid, stream)
                   : launch_scan_bf16_d1(npl, lpc, mode, a, maps, grid, stream);
}

// States per thread for `lpc` threads per channel: the smallest of 4, 8, 16
// that covers N with a kernel built for it; 0 if none does.
int npl_for(int dtype, int N, int lpc) {
  ScanVariant v;
  for (int npl : {4, 8, 16})
    if (npl * lpc >= N && variant_for(dtype, npl, lpc, &v)) return npl;
  return 0;
}

// Plan choice, from sweeps of the scan on B300 (bf16, N = 16):
//  - with at least 8 resident warps per SM of channels (B * D >= 256 per SM),
//    one lane per channel and no time split is fastest: the fewest
//    instructions per state and no aggregate pass;
//  - long sequences (L >= kLongSeq) with fewer channels split time into
//    segments of at least kMinSegSteps steps, one lane per channel, aiming at
//    32 warps per SM: the aggregate pass costs about 0.6 of a full pass over
//    the same steps, less than the lane-sharing overhead and the idle SMs it
//    replaces;
//  - otherwise the states of a channel are spread over up to 4 lanes to
//    reach 8 warps per SM;
//  - then, if fewer than 2 CTAs per SM result, time is split into segments of
//    at least kMinSegSteps steps, aiming at 8 CTAs per SM (at most 64
//    segments). Batch-1 prefill shapes on B300 (L 2048: B1 x D 1536 / 2560 /
//    5120) ran in 60 / 89 / 151 us with 8 segments, against 84 / 103 / 195 us
//    with the 4 / 4 / 2 segments of a 256-threads-per-SM target and
//    512-step minimum; B1 D1536 L8192 ran in 200 us with 32 segments against
//    257 us with 16. Layers with 2 or more CTAs per SM (the 130M- and
//    1.4B-shaped ones) stay unsplit: a split adds an aggregate pass and a
//    second wave.
constexpr int kTargetThreadsPerSM = 256;
constexpr int kSplitTargetCtasPerSM = 8;
constexpr int kLongSeq = 8192;
constexpr int kMinSegSteps = 256;

struct Plan {
  int npl, lpc, cb, nseg, seg_len, chunk;
  int tl;  // time lanes per channel (1: the sequential walk)
  bool tma_x, tma_bc;
};

constexpr int kTpChunk = 16;  // chunk of the time-parallel scan

mamba_status_t make_plan(int dtype, int batch, int dim, int N, int L, const mamba_scan_plan_t* knobs, int sms,
                         const void* u, const void* delta, const void* z, const void* Bp, const void* Cp,
                         Plan* plan) {
  const int es = dtype == 0 ? 4 : 2;
  const int tl = knobs ? std::max(1, knobs->time_lanes) : 1;
  if (tl > 1) {
    // The time-parallel chunk scan: one segment, all states of a channel per lane.
    if (N > 16) return fail(MAMBA_ERR_UNSUPPORTED, "time_lanes=%d needs dstate <= 16 (got %d)", tl, N);
    if (knobs->discretization != 0)
      return fail(MAMBA_ERR_UNSUPPORTED, "time_lanes=%d is built for the zero-order hold only", tl);
    if (knobs->segments > 1 || knobs->lanes_per_channel > 1)
      return fail(MAMBA_ERR_INVALID_ARG, "time_lanes=%d takes segments and lanes_per_channel 0 or 1", tl);
    const int cb = kScanThreads / tl;
    const bool x_ok = ((long long)dim * es) % 16 == 0 && aligned16(u) && aligned16(delta) &&
                      (!z || aligned16(z)) && (cb * es) % 16 == 0;
    const bool bc_ok = ((long long)N * es) % 16 == 0 && aligned16(Bp) && aligned16(Cp);
    if (knobs->use_tma == 1 && !(x_ok && bc_ok))
      return fail(MAMBA_ERR_INVALID_ARG, "use_tma=1 but the layout does not allow TMA tiles");
    plan->npl = 16;
    plan->lpc = 1;
    plan->tl = tl;
    plan->cb = cb;
    plan->nseg = 1;
    plan->seg_len = L;
    plan->chunk = kTpChunk;
    plan->tma_x = knobs->use_tma != 2 && x_ok;
    plan->tma_bc = knobs->use_tma != 2 && bc_ok;
    return MAMBA_OK;
  }
  int lpc_min = 1;
  while (lpc_min * 16 < N) lpc_min *= 2;
  int lpc = knobs ? knobs->lanes_per_channel : 0;
  int nseg = knobs ? knobs->segments : 0;
  const long long channels = (long long)batch * dim;
  const long long target = (long long)sms * kTargetThreadsPerSM;
  const bool long_split = channels * lpc_min < target && L >= kLongSeq;
  if (lpc == 0) {
    lpc = lpc_min;
    if (!long_split) {
      // Spread a channel's states over more threads while that is needed to
      // fill the device, up to 4 lanes and at least 4 real states per lane.
      while (channels * lpc < target && lpc * 2 <= std::max(4, lpc_min) && N >= 4 * lpc * 2 &&
             npl_for(dtype, N, lpc * 2) != 0)
        lpc *= 2;
    }
  }
  if (lpc < lpc_min || (lpc & (lpc - 1)) != 0 || lpc > 16)
    return fail(MAMBA_ERR_INVALID_ARG, "lanes_per_channel=%d is not a power of two in [%d, 16] for N=%d", lpc,
                lpc_min, N);
  const int npl = npl_for(dtype, N, lpc);
  ScanVariant v;
  if (npl == 0 || !variant_for(dtype, npl, lpc, &v))
    return fail(MAMBA_ERR_UNSUPPORTED, "no scan kernel for N=%d with lanes_per_channel=%d", N, lpc);

  const int max_seg = std::max(1, std::min(65535, (L + v.chunk - 1) / v.chunk));
  if (nseg == 0) {
    const long long ctas = ((long long)dim + v.cb - 1) / v.cb * batch;
    const long long want = (long long)sms * kSplitTargetCtasPerSM;
    nseg = 1;
    // rounded down, so that the split fills at most the waves aimed at
    // (long sequence, 40 channel blocks: 29 segments, 1,160 CTAs for 1,184
    // slots, ran in 1.66 ms against 1.70 ms with 30 segments, 1,200 CTAs)
    if (ctas < 2LL * sms) nseg = int(std::max(1LL, want / ctas));
    // segments of at least kMinSegSteps steps, at most 64 segments
    nseg = std::min({nseg, 64, std::max(1, L / kMinSegSteps)});
  }
  if (nseg < 1) return fail(MAMBA_ERR_INVALID_ARG, "segments=%d must be >= 1", nseg);
  nseg = std::min(nseg, max_seg);
  int seg_len = (L + nseg - 1) / nseg;
  seg_len = (seg_len + v.chunk - 1) / v.chunk * v.chunk;
  nseg = (L + seg_len - 1) / seg_len;  // every segment non-empty

  const bool x_ok = ((long long)dim * es) % 16 == 0 && aligned16(u) && aligned16(delta) && (!z || aligned16(z)) &&
                    (v.cb * es) % 16 == 0;
  const bool bc_ok = ((long long)N * es) % 16 == 0 && aligned16(Bp) && aligned16(Cp);
  const int use_tma = knobs ? knobs->use_tma : 0;
  if (use_tma == 1 && !(x_ok && bc_ok))
    return fail(MAMBA_ERR_INVALID_ARG,
                "use_tma=1 but the layout does not allow TMA tiles (needs 16-byte aligned pointers, "
                "dim*%d and dstate*%d multiples of 16 bytes)", es, es);
  plan->npl = npl;
  plan->lpc = lpc;
  plan->tl = 1;
  plan->cb = v.cb;
  plan->nseg = nseg;
  plan->seg_len = seg_len;
  plan->chunk = v.chunk;
  plan->tma_x = use_tma != 2 && x_ok;
  plan->tma_bc = use_tma != 2 && bc_ok;
  return MAMBA_OK;
}

// Wait limit (ns) the next scan and decode launches give their first
// mbarrier waits; mamba_set_wait_limit_ns changes it (a test setting).
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNsDefault};

// The scan entry points' common body. conv_w == nullptr: u is the scan input;
// otherwise u holds the conv input x and the kernels compute
// u = SiLU(causal conv1d(x; conv_w, conv_b)) on the fly.
//
// static_scratch: NULL for the regular entry points, whose split-sequence
// workspace comes from cudaMallocAsync on the call's stream; otherwise the
// device address of a static array of static_bytes bytes that the workspace
// must fit in (the allocation-free entry point), and nothing is allocated.
mamba_status_t scan_fwd_impl(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype, const void* u,
                             const void* delta, const float* A_log, const void* B, const void* C, const float* D,
                             const void* z, const float* delta_bias, const float* initial_state, void* out,
                             float* last_state, const mamba_scan_plan_t* plan_knobs, mamba_stream_t stream_,
                             const float* conv_w, const float* conv_b, int conv_width, float* static_scratch = nullptr,
                             size_t static_bytes = 0) {
  t_detail.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 0 || dim < 0 || seqlen < 0)
    return fail(MAMBA_ERR_INVALID_ARG, "negative size (batch=%d dim=%d seqlen=%d)", batch, dim, seqlen);
  if (dstate < 1) return fail(MAMBA_ERR_INVALID_ARG, "dstate=%d must be >= 1", dstate);
  if (dstate > kMaxState) return fail(MAMBA_ERR_UNSUPPORTED, "dstate=%d exceeds %d", dstate, kMaxState);
  if (in_dtype != MAMBA_F32 && in_dtype != MAMBA_BF16)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown in_dtype %d", int(in_dtype));
  if (batch > 65535) return fail(MAMBA_ERR_UNSUPPORTED, "batch=%d exceeds 65535", batch);
  if (plan_knobs && (plan_knobs->lanes_per_channel < 0 || plan_knobs->segments < 0 || plan_knobs->use_tma < 0 ||
                     plan_knobs->use_tma > 2 || plan_knobs->discretization < 0 || plan_knobs->discretization > 1 ||
                     (plan_knobs->time_lanes != 0 && plan_knobs->time_lanes != 1 && plan_knobs->time_lanes != 2 &&
                      plan_knobs->time_lanes != 4)))
    return fail(MAMBA_ERR_INVALID_ARG, "negative or unknown plan knob");
  const int disc = plan_knobs ? plan_knobs->discretization : 0;
  if (conv_w && (conv_width < 1 || conv_width > 4))
    return fail(MAMBA_ERR_UNSUPPORTED, "conv_width=%d must be 1..4", conv_width);
  if (conv_w && disc != 0)
    return fail(MAMBA_ERR_UNSUPPORTED, "the fused conv1d is built for the zero-order-hold discretisation only");
  if (conv_w && plan_knobs && plan_knobs->time_lanes > 1)
    return fail(MAMBA_ERR_UNSUPPORTED, "the fused conv1d is not built with time_lanes > 1");
  if (batch == 0 || dim == 0) return MAMBA_OK;
  const int dtype = in_dtype == MAMBA_F32 ? 0 : 1;
  const size_t es = dtype == 0 ? 4 : 2;
  const size_t n_state = (size_t)batch * dim * dstate;
  if (!A_log) return fail(MAMBA_ERR_INVALID_ARG, "A_log is NULL");
  if (seqlen == 0) {
    if (last_state) {
      cudaError_t e = initial_state
                          ? cudaMemcpyAsync(last_state, initial_state, n_state * 4, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(last_state, 0, n_state * 4, stream);
      if (e != cudaSuccess) return cuda_fail(e, "empty-sequence last_state");
    }
    return MAMBA_OK;
  }
  if (!u || !delta || !B || !C || !out)
    return fail(MAMBA_ERR_INVALID_ARG, "a required pointer is NULL (u=%p delta=%p B=%p C=%p out=%p)", u, delta, B, C,
                out);
  const size_t nx = (size_t)batch * seqlen * dim * es;
  const size_t nbc = (size_t)batch * seqlen * dstate * es;
  const void* inputs[] = {u, delta, z, B, C, A_log, D, delta_bias, initial_state, conv_w, conv_b};
  const size_t sizes[] = {nx, nx, nx, nbc, nbc, (size_t)dim * dstate * 4, (size_t)dim * 4, (size_t)dim * 4,
                          n_state * 4, (size_t)dim * (conv_w ? conv_width : 0) * 4, (size_t)dim * 4};
  for (int i = 0; i < 11; ++i) {
    if (overlaps(out, nx, inputs[i], sizes[i])) return fail(MAMBA_ERR_INVALID_ARG, "out aliases input %d", i);
    if (overlaps(last_state, n_state * 4, inputs[i], sizes[i]))
      return fail(MAMBA_ERR_INVALID_ARG, "last_state aliases input %d", i);
  }
  if (overlaps(out, nx, last_state, n_state * 4)) return fail(MAMBA_ERR_INVALID_ARG, "out aliases last_state");

  DeviceInfo di;
  mamba_status_t st = device_info(&di);
  if (st != MAMBA_OK) return st;
  Plan plan;
  st = make_plan(dtype, batch, dim, dstate, seqlen, plan_knobs, di.sms, u, delta, z, B, C, &plan);
  if (st != MAMBA_OK) return st;

  const size_t ws_rows = (size_t)batch * (plan.nseg - 1) * dim;
  const size_t ws_bytes = ws_rows * (dstate + 1) * sizeof(float);
  if (static_scratch && ws_bytes > static_bytes)
    return fail(MAMBA_ERR_UNSUPPORTED,
                "the plan (%d segments) needs %zu bytes of scratch; the static scratch holds %zu bytes "
                "(use fewer segments)", plan.nseg, ws_bytes, static_bytes);

  ScanMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const uint32_t cb = uint32_t(plan.cb);
  if (plan.tma_x) {
    const uint32_t urows = plan.chunk + (conv_w ? 3 : 0);  // the fused conv reads 3 steps before the chunk
    if ((st = encode_3d(&maps.u, u, int(es), dim, seqlen, batch, cb, urows)) != MAMBA_OK) return st;
    if ((st = encode_3d(&maps.delta, delta, int(es), dim, seqlen, batch, cb, plan.chunk)) != MAMBA_OK) return st;
    if (z && (st = encode_3d(&maps.z, z, int(es), dim, seqlen, batch, cb, plan.chunk)) != MAMBA_OK) return st;
  }
  if (plan.tma_bc) {
    if ((st = encode_3d(&maps.B, B, int(es), dstate, seqlen, batch, dstate, plan.chunk)) != MAMBA_OK) return st;
    if ((st = encode_3d(&maps.C, C, int(es), dstate, seqlen, batch, dstate, plan.chunk)) != MAMBA_OK) return st;
  }

  ScanArgs a;
  std::memset(&a, 0, sizeof(a));
  a.batch = batch;
  a.dim = dim;
  a.dstate = dstate;
  a.seqlen = seqlen;
  a.nseg = plan.nseg;
  a.seg_len = plan.seg_len;
  a.u = u;
  a.delta = delta;
  a.z = z;
  a.B = B;
  a.C = C;
  a.A_log = A_log;
  a.D = D;
  a.delta_bias = delta_bias;
  a.h0 = initial_state;
  a.out = out;
  a.last_state = last_state;
  a.tma_x = plan.tma_x;
  a.tma_bc = plan.tma_bc;
  a.status = di.status;
  a.conv_w = conv_w;
  a.conv_b = conv_w ? conv_b : nullptr;
  a.conv_width = conv_w ? conv_width : 0;
  a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);

  auto launch = [&](ScanMode mode, unsigned nz) {
    dim3 grid((dim + cb - 1) / cb, batch, nz);
    if (plan.tl > 1) return launch_scan_tp(dtype, plan.tl, a, maps, grid, stream);
    return launch_scan_pass(dtype, disc, plan.npl, plan.lpc, mode, a, maps, grid, stream);
  };

  void* work = nullptr;  // the workspace when it is allocated here
  if (plan.nseg > 1) {
    float* ws = static_scratch;  // every value is written by the aggregate pass before the full pass reads it
    if (!ws) {
      cudaError_t e = cudaMallocAsync(&work, ws_bytes, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(split-sequence workspace)");
      ws = static_cast<float*>(work);
    }
    a.agg_h = ws;
    a.agg_dsum = ws + ws_rows * dstate;
    cudaError_t e = launch(ScanMode::kAggregate, plan.nseg - 1);
    if (e != cudaSuccess) {
      if (work) cudaFreeAsync(work, stream);
      return cuda_fail(e, "scan aggregate pass launch");
    }
  }
  a.after_agg = plan.nseg > 1 ? 1 : 0;
  cudaError_t e = launch(ScanMode::kFull, plan.nseg);
  if (work) {
    cudaError_t e2 = cudaFreeAsync(work, stream);
    if (e == cudaSuccess && e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync(split-sequence workspace)");
  }
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  return MAMBA_OK;
}

}  // namespace

extern "C" {

mamba_status_t mamba_selective_scan_fwd_ex(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                           const void* u, const void* delta, const float* A_log, const void* B,
                                           const void* C, const float* D, const void* z, const float* delta_bias,
                                           const float* initial_state, void* out, float* last_state,
                                           const mamba_scan_plan_t* plan_knobs, mamba_stream_t stream) {
  return scan_fwd_impl(batch, dim, dstate, seqlen, in_dtype, u, delta, A_log, B, C, D, z, delta_bias,
                       initial_state, out, last_state, plan_knobs, stream, nullptr, nullptr, 0);
}

mamba_status_t mamba_conv1d_selective_scan_fwd(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                               const void* x, const float* conv_weight, const float* conv_bias,
                                               int conv_width, const void* delta, const float* A_log,
                                               const void* B, const void* C, const float* D, const void* z,
                                               const float* delta_bias, const float* initial_state, void* out,
                                               float* last_state, const mamba_scan_plan_t* plan,
                                               mamba_stream_t stream) {
  if (!conv_weight && batch > 0 && dim > 0) {
    t_detail.clear();
    return fail(MAMBA_ERR_INVALID_ARG, "conv_weight is NULL");
  }
  return scan_fwd_impl(batch, dim, dstate, seqlen, in_dtype, x, delta, A_log, B, C, D, z, delta_bias,
                       initial_state, out, last_state, plan, stream, conv_weight ? conv_weight : nullptr, conv_bias,
                       conv_width);
}

mamba_status_t mamba_selective_scan_plan(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                         const mamba_scan_plan_t* knobs, mamba_scan_plan_t* chosen,
                                         int* kernel_launches) {
  t_detail.clear();
  if (!chosen || !kernel_launches) return fail(MAMBA_ERR_INVALID_ARG, "chosen / kernel_launches is NULL");
  if (batch <= 0 || dim <= 0 || seqlen <= 0)
    return fail(MAMBA_ERR_INVALID_ARG, "sizes must be positive (batch=%d dim=%d seqlen=%d)", batch, dim, seqlen);
  if (dstate < 1) return fail(MAMBA_ERR_INVALID_ARG, "dstate=%d must be >= 1", dstate);
  if (dstate > kMaxState) return fail(MAMBA_ERR_UNSUPPORTED, "dstate=%d exceeds %d", dstate, kMaxState);
  if (in_dtype != MAMBA_F32 && in_dtype != MAMBA_BF16)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown in_dtype %d", int(in_dtype));
  DeviceInfo di;
  mamba_status_t st = device_info(&di);
  if (st != MAMBA_OK) return st;
  Plan plan;
  const void* aligned = reinterpret_cast<const void*>(uintptr_t(256));
  st = make_plan(in_dtype == MAMBA_F32 ? 0 : 1, batch, dim, dstate, seqlen, knobs, di.sms, aligned, aligned,
                 aligned, aligned, aligned, &plan);
  if (st != MAMBA_OK) return st;
  chosen->lanes_per_channel = plan.lpc;
  chosen->segments = plan.nseg;
  chosen->discretization = knobs ? knobs->discretization : 0;
  chosen->time_lanes = plan.tl;
  chosen->use_tma = (plan.tma_x && plan.tma_bc) ? 1 : 2;
  *kernel_launches = plan.nseg > 1 ? 2 : 1;
  return MAMBA_OK;
}

mamba_status_t mamba_selective_scan_fwd(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                        const void* u, const void* delta, const float* A_log, const void* B,
                                        const void* C, const float* D, const void* z, const float* delta_bias,
                                        void* out, float* last_state, mamba_stream_t stream) {
  return mamba_selective_scan_fwd_ex(batch, dim, dstate, seqlen, in_dtype, u, delta, A_log, B, C, D, z, delta_bias,
                                     nullptr, out, last_state, nullptr, stream);
}

mamba_status_t mamba_selective_state_update_ex(int batch, int dim, int dstate, mamba_dtype_t in_dtype,
                                               float* state, const void* u, const void* delta, const float* A_log,
                                               const void* B, const void* C, const float* D, const void* z,
                                               const float* delta_bias, void* out, int discretization,
                                               mamba_stream_t stream_) {
  t_detail.clear();
  if (discretization < 0 || discretization > 1)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown discretization %d", discretization);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 0 || dim < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (batch=%d dim=%d)", batch, dim);
  if (dstate < 1) return fail(MAMBA_ERR_INVALID_ARG, "dstate=%d must be >= 1", dstate);
  if (dstate > kMaxState) return fail(MAMBA_ERR_UNSUPPORTED, "dstate=%d exceeds %d", dstate, kMaxState);
  if (in_dtype != MAMBA_F32 && in_dtype != MAMBA_BF16)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown in_dtype %d", int(in_dtype));
  if (batch > 4 * 65535) return fail(MAMBA_ERR_UNSUPPORTED, "batch=%d exceeds %d", batch, 4 * 65535);
  if (batch == 0 || dim == 0) return MAMBA_OK;
  if (!state || !u || !delta || !A_log || !B || !C || !out)
    return fail(MAMBA_ERR_INVALID_ARG, "a required pointer is NULL");
  const size_t es = in_dtype == MAMBA_F32 ? 4 : 2;
  const size_t ns = (size_t)batch * dim * dstate * 4;
  const size_t nx = (size_t)batch * dim * es;
  const size_t nbc = (size_t)batch * dstate * es;
  const void* others[] = {u, delta, z, B, C, A_log, D, delta_bias, out};
  const size_t sizes[] = {nx, nx, nx, nbc, nbc, (size_t)dim * dstate * 4, (size_t)dim * 4, (size_t)dim * 4, nx};
  for (int i = 0; i < 9; ++i)
    if (overlaps(state, ns, others[i], sizes[i])) return fail(MAMBA_ERR_INVALID_ARG, "state aliases argument %d", i);
  for (int i = 0; i < 8; ++i)
    if (overlaps(out, nx, others[i], sizes[i])) return fail(MAMBA_ERR_INVALID_ARG, "out aliases input %d", i);
  DecodeArgs a;
  a.batch = batch;
  a.dim = dim;
  a.dstate = dstate;
  a.state = state;
  a.u = u;
  a.delta = delta;
  a.z = z;
  a.B = B;
  a.C = C;
  a.A_log = A_log;
  a.D = D;
  a.delta_bias = delta_bias;
  a.out = out;
  a.disc = discretization;
  DeviceInfo di;
  const mamba_status_t st = device_info(&di);
  if (st != MAMBA_OK) return st;
  a.status = di.status;
  a.sms = di.sms;
  a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  cudaError_t e = launch_state_update(in_dtype == MAMBA_F32 ? 0 : 1, a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "state update launch");
  return MAMBA_OK;
}

mamba_status_t mamba_selective_state_update(int batch, int dim, int dstate, mamba_dtype_t in_dtype, float* state,
                                            const void* u, const void* delta, const float* A_log, const void* B,
                                            const void* C, const float* D, const void* z, const float* delta_bias,
                                            void* out, mamba_stream_t stream) {
  return mamba_selective_state_update_ex(batch, dim, dstate, in_dtype, state, u, delta, A_log, B, C, D, z,
                                         delta_bias, out, 0, stream);
}

mamba_status_t mamba_selective_scan_bwd_ex(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                           int discretization, const void* u, const void* delta, const float* A_log,
                                           const void* B, const void* C, const float* D, const void* z,
                                           const float* delta_bias, const float* initial_state, const void* dout,
                                           const float* dlast_state, void* du, void* ddelta, float* dA_log, float* dB,
                                           float* dC, float* dD, void* dz, float* ddelta_bias,
                                           float* dinitial_state, int segments, mamba_stream_t stream_) {
  t_detail.clear();
  if (segments < 0) return fail(MAMBA_ERR_INVALID_ARG, "segments=%d must be >= 0 (0 = automatic)", segments);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 0 || dim < 0 || seqlen < 0)
    return fail(MAMBA_ERR_INVALID_ARG, "negative size (batch=%d dim=%d seqlen=%d)", batch, dim, seqlen);
  if (dstate < 1) return fail(MAMBA_ERR_INVALID_ARG, "dstate=%d must be >= 1", dstate);
  if (in_dtype != MAMBA_F32 && in_dtype != MAMBA_BF16)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown in_dtype %d", int(in_dtype));
  if (discretization < 0 || discretization > 1)
    return fail(MAMBA_ERR_INVALID_ARG, "unknown discretization %d", discretization);
  if (!scan_bwd_supported(dstate))
    return fail(MAMBA_ERR_UNSUPPORTED, "the backward scan is built for dstate 16, 32, 64 or 128 (got %d)", dstate);
  if (batch > 65535) return fail(MAMBA_ERR_UNSUPPORTED, "batch=%d exceeds 65535", batch);
  if (!z && dz) return fail(MAMBA_ERR_INVALID_ARG, "dz given without z");
  if (dim > 0 && (!A_log || !dA_log)) return fail(MAMBA_ERR_INVALID_ARG, "A_log and dA_log are required");
  const bool work = batch > 0 && dim > 0 && seqlen > 0;
  if (work && (!u || !delta || !B || !C || !dout || !du || !ddelta || !dB || !dC))
    return fail(MAMBA_ERR_INVALID_ARG, "a required pointer is NULL");
  const float* f4[] = {initial_state, dlast_state, dA_log, dB, dC, dinitial_state};
  for (const float* p : f4)
    if (p && !aligned16(p))
      return fail(MAMBA_ERR_UNSUPPORTED, "fp32 state / gradient arrays must be 16-byte aligned (%p)", (const void*)p);

  const int dtype = in_dtype == MAMBA_F32 ? 0 : 1;
  const size_t es = dtype == 0 ? 4 : 2;
  const size_t nx = (size_t)batch * seqlen * dim * es;
  const size_t nbc = (size_t)batch * seqlen * dstate * es;
  const size_t nbc32 = (size_t)batch * seqlen * dstate * 4;
  const size_t ns = (size_t)batch * dim * dstate * 4;
  const size_t np = (size_t)dim * dstate * 4, nd = (size_t)dim * 4;
  const void* ins[] = {u, delta, A_log, B, C, D, z, delta_bias, initial_state, dout, dlast_state};
  const size_t in_sz[] = {nx, nx, np, nbc, nbc, nd, nx, nd, ns, nx, ns};
  void* outs[] = {du, ddelta, dA_log, dB, dC, dD, dz, ddelta_bias, dinitial_state};
  const size_t out_sz[] = {nx, nx, np, nbc32, nbc32, nd, nx, nd, ns};
  for (int i = 0; i < 9; ++i) {
    for (int j = 0; j < 11; ++j)
      if (overlaps(outs[i], out_sz[i], ins[j], in_sz[j]))
        return fail(MAMBA_ERR_INVALID_ARG, "output %d aliases input %d", i, j);
    for (int j = 0; j < i; ++j)
      if (overlaps(outs[i], out_sz[i], outs[j], out_sz[j]))
        return fail(MAMBA_ERR_INVALID_ARG, "output %d aliases output %d", i, j);
  }

  // Sums start from zero.
  cudaError_t e = cudaSuccess;
  if (dim > 0) e = cudaMemsetAsync(dA_log, 0, np, stream);
  if (e == cudaSuccess && dD && dim > 0) e = cudaMemsetAsync(dD, 0, nd, stream);
  if (e == cudaSuccess && ddelta_bias && dim > 0) e = cudaMemsetAsync(ddelta_bias, 0, nd, stream);
  if (e == cudaSuccess && nbc32 > 0) e = cudaMemsetAsync(dB, 0, nbc32, stream);
  if (e == cudaSuccess && nbc32 > 0) e = cudaMemsetAsync(dC, 0, nbc32, stream);
  if (e != cudaSuccess) return cuda_fail(e, "zeroing the gradient sums");
  if (batch == 0 || dim == 0) return MAMBA_OK;
  if (seqlen == 0) {  // last_state = initial_state
    if (dinitial_state) {
      e = dlast_state ? cudaMemcpyAsync(dinitial_state, dlast_state, ns, cudaMemcpyDeviceToDevice, stream)
                      : cudaMemsetAsync(dinitial_state, 0, ns, stream);
      if (e != cudaSuccess) return cuda_fail(e, "empty-sequence dinitial_state");
    }
    return MAMBA_OK;
  }

  // 16-byte slots when every (B, L, D) / (B, L, N) tensor allows them.
  const int cb = kBwdThreads / (dstate / 4);
  const size_t sbx = std::min<size_t>(16, (size_t)cb * es);
  bool aligned = ((size_t)dim * es) % sbx == 0;
  const void* xs[] = {u, delta, z, dout, du, ddelta, dz, B, C};
  for (const void* p : xs)
    if (p && !aligned16(p)) aligned = false;

  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.batch = batch;
  a.dim = dim;
  a.dstate = dstate;
  a.seqlen = seqlen;
  a.nchunk = (seqlen + kBwdChunk - 1) / kBwdChunk;
  a.u = u;
  a.delta = delta;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dout = dout;
  a.A_log = A_log;
  a.D = D;
  a.delta_bias = delta_bias;
  a.h0 = initial_state;
  a.dlast = dlast_state;
  a.du = du;
  a.ddelta = ddelta;
  a.dz = dz;
  a.dA_log = dA_log;
  a.dB = dB;
  a.dC = dC;
  a.dD = dD;
  a.ddelta_bias = ddelta_bias;
  a.dh0 = dinitial_state;
  a.disc = discretization;
  a.aligned = aligned ? 1 : 0;

  // Time segments: when the channel blocks x batch rows leave SMs idle, cut the sequence
  // into segments of whole chunks so that about 12 CTAs per SM are launched, keeping at
  // least 4 chunks per segment. On B300 (B1 D5120 N16 L32768, bf16) 1, 2, 5, 11 and 32
  // segments took 12.97, 10.85, 8.87, 8.11 and 8.18 ms; past about 8 the kernel runs at
  // the throughput of a full GPU and the two segment passes take the rest.
  DeviceInfo di;
  mamba_status_t st = device_info(&di);
  if (st != MAMBA_OK) return st;
  int nseg = segments;
  if (nseg == 0) {
    const long ctas = (long)((dim + cb - 1) / cb) * batch;
    nseg = 1;
    if (ctas < 2L * di.sms) nseg = int(std::min<long>(12L * di.sms / ctas, a.nchunk / 4));
  }
  nseg = std::max(1, std::min({nseg, kBwdMaxSegments, a.nchunk}));
  const int chunks_per_seg = (a.nchunk + nseg - 1) / nseg;
  a.seg_len = chunks_per_seg * kBwdChunk;
  a.nseg = (seqlen + a.seg_len - 1) / a.seg_len;

  const size_t ck_elems = (size_t)batch * a.nchunk * dim * dstate;
  const size_t seg_state = a.nseg > 1 ? (size_t)batch * a.nseg * dim * dstate : 0;
  const size_t seg_vec = a.nseg > 1 ? (size_t)batch * a.nseg * dim : 0;
  void* ck = nullptr;
  e = cudaMallocAsync(&ck, (ck_elems + 2 * seg_state + seg_vec) * sizeof(float), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(backward checkpoint workspace)");
  a.ck = static_cast<float*>(ck);
  if (a.nseg > 1) {
    a.seg_h = a.ck + ck_elems;
    a.seg_g = a.seg_h + seg_state;
    a.seg_dsum = a.seg_g + seg_state;
  }
  e = launch_scan_bwd(dtype, a, stream);
  cudaError_t e2 = cudaFreeAsync(ck, stream);
  if (e != cudaSuccess) return cuda_fail(e, "backward scan launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync(backward checkpoint workspace)");
  return MAMBA_OK;
}

mamba_status_t mamba_selective_scan_bwd(int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype,
                                        int discretization, const void* u, const void* delta, const float* A_log,
                                        const void* B, const void* C, const float* D, const void* z,
                                        const float* delta_bias, const float* initial_state, const void* dout,
                                        const float* dlast_state, void* du, void* ddelta, float* dA_log, float* dB,
                                        float* dC, float* dD, void* dz, float* ddelta_bias, float* dinitial_state,
                                        mamba_stream_t stream) {
  return mamba_selective_scan_bwd_ex(batch, dim, dstate, seqlen, in_dtype, discretization, u, delta, A_log, B, C, D,
                                     z, delta_bias, initial_state, dout, dlast_state, du, ddelta, dA_log, dB, dC, dD,
                                     dz, ddelta_bias, dinitial_state, 0, stream);
}

const char* mamba_status_string(mamba_status_t s) {
  switch (s) {
    case MAMBA_OK: return "ok";
    case MAMBA_ERR_INVALID_ARG: return "invalid argument";
    case MAMBA_ERR_UNSUPPORTED: return "unsupported";
    case MAMBA_ERR_CUDA: return "CUDA error";
    case MAMBA_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

const char* mamba_last_error_detail(void) { return t_detail.c_str(); }

mamba_status_t mamba_device_status(int* status_out, mamba_stream_t stream_) {
  t_detail.clear();
  if (!status_out) return fail(MAMBA_ERR_INVALID_ARG, "status_out is NULL");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  DeviceInfo di;
  mamba_status_t st = device_info(&di);
  if (st != MAMBA_OK) return st;
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, di.status, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(di.status, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *status_out = word;
  return MAMBA_OK;
}

int mamba_version(void) { return kVersion; }

unsigned long long mamba_set_wait_limit_ns(unsigned long long limit_ns) {
  return g_wait_limit_ns.exchange(limit_ns);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free scan entry point: the split-sequence workspace lives in a
// static device array instead of a cudaMallocAsync allocation.
static __device__ __align__(256) float g_noalloc_scratch[MAMBA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Looks the array's device address up once per device, with that device current.
mamba_status_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MAMBA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    float* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scan scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MAMBA_OK;
}
}  // namespace

extern "C" mamba_status_t mamba_selective_scan_fwd_noalloc(
    int batch, int dim, int dstate, int seqlen, mamba_dtype_t in_dtype, const void* u, const void* delta,
    const float* A_log, const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
    const float* initial_state, void* out, float* last_state, const mamba_scan_plan_t* plan_knobs,
    mamba_stream_t stream) {
  t_detail.clear();
  float* scratch = nullptr;
  const mamba_status_t st = noalloc_scratch(&scratch);
  if (st != MAMBA_OK) return st;
  return scan_fwd_impl(batch, dim, dstate, seqlen, in_dtype, u, delta, A_log, B, C, D, z, delta_bias, initial_state,
                       out, last_state, plan_knobs, stream, nullptr, nullptr, 0, scratch,
                       MAMBA_NOALLOC_SCRATCH_BYTES);
}
