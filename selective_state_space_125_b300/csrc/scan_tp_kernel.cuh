// Time-parallel selective scan within each chunk (plan knob time_lanes).
//
// The operator form of the recurrence ("State Space Models and Mamba" §4,
// parallel scan; "Mamba" paper notes, Design 2; x-humanoid CSDN §2.2: the
// chunk is scanned in parallel on chip and the state passed between chunks):
// a run of steps acts on the state as h -> a h + b, with a = prod Abar and b
// the state the run reaches from zero, and consecutive runs compose as
//   (a, b) o (a', b') = (a a', a' b + b').
// Because A is constant in time, the a of a run is exp(A sum dt), one scalar
// sum per channel.
//
// Work layout: TL consecutive lanes share one channel and hold all of its
// N <= 16 states; a chunk of 16 steps is cut into TL runs of S = 16 / TL
// steps, one per lane. Per chunk, each lane:
//   1. scans its run sequentially (lane 0 from the chunk's carry-in state,
//      the others from zero), keeping each step's partial readout;
//   2. takes part in a Hillis-Steele scan of the runs' (sum dt, end state)
//      over the TL lanes by warp shuffles, composed with the operator above,
//      which gives every lane the exact state entering its run and the chunk's
//      end state (the next chunk's carry);
//   3. fixes its readouts up with the state entering its run, decayed step by
//      step over the run (sum_n C_n (prod Abar) h_in,n), then applies the D
//      skip and the SiLU gate and stores its S outputs.
// Against the sequential walk of scan_kernel this adds the scan of step 2
// and the fix-up of step 3 (about two thirds of a step's arithmetic per
// step), in exchange for TL times the threads per channel.
//
// Staging (TMA tiles with mbarriers, or plain loads), the fast and precise
// arithmetic, the |A| floor and the optimistic fast pass with an accurate
// rerun follow scan_kernel.cuh. Zero-order hold only, N <= 16, one time
// segment; initial_state and last_state as in the other plans.
#pragma once

#include <type_traits>

#include "scan_kernel.cuh"

namespace mamba {

template <typename Tin, int TL>
struct ScanTpGeom {
  static constexpr int kNPL = 16;                 // all states of a channel (padded)
  static constexpr int kCB = kScanThreads / TL;   // channels per CTA
  static constexpr int kES = int(sizeof(Tin));
  static constexpr int kChunk = 16;
  static constexpr int kRun = kChunk / TL;        // steps per lane per chunk
  static constexpr int kStages = 3;
  static constexpr size_t kXTile = scan_a128(size_t(kChunk) * kCB * kES);
  static constexpr size_t kBCTile = scan_a128(size_t(kChunk) * kNPL * kES);
  static constexpr size_t kStage = 3 * kXTile + 2 * kBCTile;  // u, delta, z, B, C
  static constexpr size_t kBC32 = scan_a128(size_t(kChunk) * 2 * kNPL * 4);
  static constexpr size_t kChan = scan_a128(size_t(kCB) * 2 * 4);
  static constexpr size_t kSave = scan_a128(size_t(kScanThreads) * kNPL * 4);
  static constexpr size_t kRunBuf = scan_a128(size_t(kRun) * kScanThreads * 4);  // per-step values of my run
  static constexpr size_t kOffBC32 = kStages * kStage;
  static constexpr size_t kOffChan = kOffBC32 + 2 * kBC32;
  static constexpr size_t kOffSave = kOffChan + kChan;
  static constexpr size_t kOffRunY = kOffSave + kSave;
  static constexpr size_t kOffRunDt = kOffRunY + kRunBuf;
  static constexpr size_t kOffBar = kOffRunDt + kRunBuf;
  static constexpr size_t kSmem = kOffBar + 128 + 128;
  static_assert(kChunk % TL == 0 && TL >= 2 && TL <= 8, "runs of whole steps");
  static_assert(kSmem <= 227 * 1024, "time-parallel scan exceeds the shared memory of one CTA");
};

template <typename Tin, int TL>
__global__ void __launch_bounds__(kScanThreads, 3)
    scan_tp_kernel(const ScanArgs a, const __grid_constant__ ScanMaps maps) {
  using G = ScanTpGeom<Tin, TL>;
  using E = Elem<Tin>;
  constexpr bool PRECISE = std::is_same<Tin, float>::value;
  constexpr int CB = G::kCB, CH = G::kChunk, NS = G::kStages, S = G::kRun;
  constexpr int NPL = G::kNPL, NH = NPL / 2;
  constexpr unsigned kFull = 0xffffffffu;

  extern __shared__ unsigned char smem_dyn[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  float* chan_bias = reinterpret_cast<float*>(smem + G::kOffChan);
  float* chan_D = chan_bias + CB;
  float4* save = reinterpret_cast<float4*>(smem + G::kOffSave);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + G::kOffBar);
  auto xu = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage); };
  auto xd = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kXTile); };
  auto xz = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + 2 * G::kXTile); };
  auto braw = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + 3 * G::kXTile); };
  auto craw = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + 3 * G::kXTile + G::kBCTile); };
  auto bc32 = [&](int k) { return reinterpret_cast<float*>(smem + G::kOffBC32 + (k & 1) * G::kBC32); };

  const int tid = threadIdx.x;
  const int c = tid / TL, q = tid % TL;
  float* run_y = reinterpret_cast<float*>(smem + G::kOffRunY) + tid;  // [step of my run][threads]
  float* run_dt = reinterpret_cast<float*>(smem + G::kOffRunDt) + tid;
  const int Dm = a.dim, N = a.dstate, L = a.seqlen;
  const int d0 = blockIdx.x * CB;
  const int d = d0 + c;
  const bool dvalid = d < Dm;
  const int b = blockIdx.y;
  const int nchunks = (L + CH - 1) / CH;
  const bool has_z = a.z != nullptr;
  const bool use_tma = a.tma_x || a.tma_bc;
  const Tin* gu = static_cast<const Tin*>(a.u);
  const Tin* gdl = static_cast<const Tin*>(a.delta);
  const Tin* gz = static_cast<const Tin*>(a.z);
  const Tin* gB = static_cast<const Tin*>(a.B);
  const Tin* gC = static_cast<const Tin*>(a.C);

  for (int i = tid; i < CB; i += kScanThreads) {
    const int dd = d0 + i;
    chan_bias[i] = (a.delta_bias && dd < Dm) ? a.delta_bias[dd] : 0.0f;
    chan_D[i] = (a.D && dd < Dm) ? a.D[dd] : 0.0f;
  }

  auto issue = [&](int k) {
    const int s = k % NS;
    const int t0 = k * CH;
    uint32_t bytes = 0;
    if (a.tma_x) bytes += uint32_t((has_z ? 3 : 2) * CH * CB * sizeof(Tin));
    if (a.tma_bc) bytes += 2u * uint32_t(CH * N * sizeof(Tin));
    mbar_arrive_expect_tx(&mbar[s], bytes);
    if (a.tma_x) {
      tma_load_3d(xu(s), &maps.u, d0, t0, b, &mbar[s]);
      tma_load_3d(xd(s), &maps.delta, d0, t0, b, &mbar[s]);
      if (has_z) tma_load_3d(xz(s), &maps.z, d0, t0, b, &mbar[s]);
    }
    if (a.tma_bc) {
      tma_load_3d(braw(s), &maps.B, 0, t0, b, &mbar[s]);
      tma_load_3d(craw(s), &maps.C, 0, t0, b, &mbar[s]);
    }
  };
  if (use_tma && tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&mbar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  int issued = 0;
  if (use_tma && tid == 0)
    for (; issued < min(NS, nchunks); ++issued) issue(issued);

  // A = -exp(A_log) (|A| >= kMinAbsA), Ak = A log2(e) (fast) or A (precise),
  // Ik = 1 / A; st: the state entering the chunk (every lane holds it).
  float2 Ak[NH], Ik[NH], st[NH];
  float minA = 3.0e38f;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const bool real = j < N;
    float A = -1.0f;
    if (dvalid && real) A = -expf(a.A_log[(size_t)d * N + j]);
    A = fminf(A, -kMinAbsA);
    if (real) minA = fminf(minA, -A);
    const float ak = real ? (PRECISE ? A : A * kLog2e) : 0.0f;
    const float ik = real ? 1.0f / A : 0.0f;
    const float hin = (dvalid && real && a.h0) ? a.h0[((size_t)b * Dm + d) * N + j] : 0.0f;
    const float sv = PRECISE ? hin : hin * A;
    if (j % 2 == 0) {
      Ak[j / 2].x = ak; Ik[j / 2].x = ik; st[j / 2].x = sv;
    } else {
      Ak[j / 2].y = ak; Ik[j / 2].y = ik; st[j / 2].y = sv;
    }
  }
  const float thr = PRECISE ? 0.0f : kFastMinDtA / minA;
  const float bias = chan_bias[c];
  const float Dd = chan_D[c];
  auto decay_of = [&](float ak, float dsum) { return PRECISE ? expf(ak * dsum) : hw_ex2(ak * dsum); };

  // One chunk (see the file comment). Returns (fast pass) whether a lane of
  // the warp met a live step with dt < thr.
  auto run_chunk = [&]<bool HZ, bool ACC>(int s, int kc, int t0, int tv) -> bool {
    const Tin* su = xu(s) + c;
    const Tin* sd = xd(s) + c;
    const Tin* sz = xz(s) + c;
    const float* bc = bc32(kc);
    const int tb = q * S;  // my run: steps tb .. tb + S - 1 of the chunk
    float dtmin = 3.0e38f;  // smallest dt met (fast pass)
    float2 sl[NH];  // my run's state: from the carry (lane 0) or from zero
#pragma unroll
    for (int j = 0; j < NH; ++j) sl[j] = q == 0 ? st[j] : make_float2(0.0f, 0.0f);
    float dsum = 0.0f;
#pragma unroll 2
    for (int i = 0; i < S; ++i) {
      const int tm = tb + i;
      const bool live = tm < tv;
      const float xm = E::load(sd + tm * CB) + bias;
      const float dtv = PRECISE ? softplus_precise(xm) : softplus_fast(xm);
      const float dt = live ? dtv : 0.0f;
      const float u = live ? E::load(su + tm * CB) : 0.0f;
      if (!PRECISE && !ACC) dtmin = fminf(dtmin, dtv);
      run_dt[i * kScanThreads] = dt;
      dsum += dt;
      const float* Bt = bc + tm * 2 * NPL;
      if constexpr (PRECISE)
        run_y[i * kScanThreads] = step_precise<NPL, true>(sl, Ak, Ik, dt, u, Bt, Bt + NPL);
      else
        run_y[i * kScanThreads] = step_fast<NPL, true, ACC>(sl, Ak, Ik, dt, u, Bt, Bt + NPL);
    }
    // Inclusive scan of the runs (sum dt, end state) over the channel's TL
    // lanes: lane q ends with the exact state after its run.
    float D = dsum;
#pragma unroll
    for (int o = 1; o < TL; o <<= 1) {
      const float Dp = __shfl_up_sync(kFull, D, o, TL);
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float px = __shfl_up_sync(kFull, sl[j].x, o, TL);
        const float py = __shfl_up_sync(kFull, sl[j].y, o, TL);
        if (q >= o) {
          sl[j].x = fmaf(decay_of(Ak[j].x, D), px, sl[j].x);
          sl[j].y = fmaf(decay_of(Ak[j].y, D), py, sl[j].y);
        }
      }
      if (q >= o) D += Dp;
    }
    // The state entering my run (lane q - 1's), and the chunk's end state.
    float2 cin[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      const float cx = __shfl_up_sync(kFull, sl[j].x, 1, TL);
      const float cy = __shfl_up_sync(kFull, sl[j].y, 1, TL);
      cin[j] = q == 0 ? make_float2(0.0f, 0.0f) : make_float2(cx, cy);
      st[j] = make_float2(__shfl_sync(kFull, sl[j].x, TL - 1, TL), __shfl_sync(kFull, sl[j].y, TL - 1, TL));
    }
    // Fix-up: add what the state entering my run contributes to each readout,
    // decayed step by step; then the D skip, the gate and the stores.
#pragma unroll 2
    for (int i = 0; i < S; ++i) {
      const int tm = tb + i;
      const float* Ct = bc + tm * 2 * NPL + NPL;
      float2 yy = make_float2(0.0f, 0.0f);
      const float dti = run_dt[i * kScanThreads];
      const float2 dd = make_float2(dti, dti);
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float2 x = __fmul2_rn(dd, Ak[j]);
        const float2 ab = PRECISE ? make_float2(expf(x.x), expf(x.y)) : make_float2(hw_ex2(x.x), hw_ex2(x.y));
        cin[j] = __fmul2_rn(ab, cin[j]);
        const float2 Cp = *reinterpret_cast<const float2*>(Ct + 2 * j);
        yy = __ffma2_rn(PRECISE ? Cp : __fmul2_rn(Cp, Ik[j]), cin[j], yy);
      }
      float y = run_y[i * kScanThreads] + (yy.x + yy.y);
      if (dvalid && tm < tv) {
        y = fmaf(Dd, E::load(su + tm * CB), y);
        if (HZ) {
          const float zf = E::load(sz + tm * CB);
          y *= PRECISE ? silu_precise(zf) : silu_fast(zf);
        }
        E::store(static_cast<Tin*>(a.out) + ((size_t)b * L + t0 + tm) * Dm + d, y);
      }
    }
    if constexpr (!PRECISE && !ACC) return __any_sync(kFull, dtmin < thr);
    return false;
  };

  for (int k = 0; k < nchunks; ++k) {
    const int s = k % NS;
    const int t0 = k * CH;
    const int tv = min(CH, L - t0);
    if (use_tma) {
      const bool ok = mbar_wait_bounded(&mbar[s], (k / NS) & 1, a.wait_ns);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          record_status(a.status, kStatusTimeout);
          for (int kk = k; kk < issued; ++kk) mbar_wait_bounded(&mbar[kk % NS], (kk / NS) & 1);
        }
        return;
      }
    }
    if (!a.tma_x) {
      for (int i = tid; i < CH * CB; i += kScanThreads) {
        const int t = i / CB, cc = i % CB;
        const int gt = t0 + t, gd = d0 + cc;
        const bool in = gt < L && gd < Dm;
        const size_t off = ((size_t)b * L + gt) * Dm + gd;
        xu(s)[i] = in ? gu[off] : Tin(0.0f);
        xd(s)[i] = in ? gdl[off] : Tin(0.0f);
        if (has_z) xz(s)[i] = in ? gz[off] : Tin(0.0f);
      }
    }
    float* bck = bc32(k);
    for (int i = tid; i < CH * NPL; i += kScanThreads) {
      const int t = i / NPL, n = i % NPL;
      float bv = 0.0f, cv = 0.0f;
      if (n < N) {
        if (a.tma_bc) {
          bv = E::load(braw(s) + t * N + n);
          cv = E::load(craw(s) + t * N + n);
        } else if (t0 + t < L) {
          const size_t off = ((size_t)b * L + t0 + t) * N + n;
          bv = E::load(gB + off);
          cv = E::load(gC + off);
        }
      }
      bck[t * 2 * NPL + n] = bv;
      bck[t * 2 * NPL + NPL + n] = cv;
    }
    __syncthreads();  // chunk k staged; every thread is past chunk k-1
    if (use_tma && tid == 0 && k >= 1 && issued < nchunks) {
      fence_proxy_async_smem();
      issue(issued);
      ++issued;
    }
    if constexpr (!PRECISE) {
#pragma unroll
      for (int j = 0; j < NH; j += 2)
        save[(j / 2) * kScanThreads + tid] = make_float4(st[j].x, st[j].y, st[j + 1].x, st[j + 1].y);
      const bool redo = has_z ? run_chunk.template operator()<true, false>(s, k, t0, tv)
                              : run_chunk.template operator()<false, false>(s, k, t0, tv);
      if (redo) {
#pragma unroll
        for (int j = 0; j < NH; j += 2) {
          const float4 v = save[(j / 2) * kScanThreads + tid];
          st[j] = make_float2(v.x, v.y);
          st[j + 1] = make_float2(v.z, v.w);
        }
        if (has_z)
          run_chunk.template operator()<true, true>(s, k, t0, tv);
        else
          run_chunk.template operator()<false, true>(s, k, t0, tv);
      }
    } else if (has_z) {
      run_chunk.template operator()<true, false>(s, k, t0, tv);
    } else {
      run_chunk.template operator()<false, false>(s, k, t0, tv);
    }
  }

  if (dvalid && q == 0 && a.last_state) {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const float sv = (j % 2 == 0) ? st[j / 2].x : st[j / 2].y;
      const float ik = (j % 2 == 0) ? Ik[j / 2].x : Ik[j / 2].y;
      if (j < N) a.last_state[((size_t)b * Dm + d) * N + j] = PRECISE ? sv : sv * ik;
    }
  }
}

template <typename Tin, int TL>
cudaError_t launch_scan_tp_variant(const ScanArgs& a, const ScanMaps& maps, dim3 grid, cudaStream_t stream) {
  using G = ScanTpGeom<Tin, TL>;
  static bool configured = false;  // per instantiation; benign race (idempotent)
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(scan_tp_kernel<Tin, TL>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(G::kSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  scan_tp_kernel<Tin, TL><<<grid, kScanThreads, G::kSmem, stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace mamba
