// Selective-scan kernels for sm_103a.
//
// Method ("State Space Models and Mamba" §2 and §4; "Mamba" paper notes,
// Design 1 and Design 2): per batch b, channel d and state n,
//   dt = softplus(delta + bias_d), Abar = exp(dt A_n), Bbar = (Abar - 1) / A_n * B_n,
//   h  = Abar h + Bbar u,  y = sum_n C_n h_n + D_d u,  out = y * SiLU(z).
// Hardware-aware in the sense of the pages' §3.3.2 remark: only u, delta, z,
// B, C are read from HBM and only out (and last_state) is written; dt, Abar,
// Bbar and h exist only in registers and shared memory.
//
// Layout of work:
//   - a CTA owns kCB = 128 / LPC channels of one batch row and one time
//     segment; LPC consecutive lanes of a warp share a channel, each holding
//     NPL of its states in registers (NPL * LPC >= N, the rest padded with
//     zeros);
//   - time is walked in chunks of kChunk steps. Thread 0 stages each chunk's
//     u / delta / z tiles ([chunk][channels]) and B / C tiles ([chunk][N])
//     into shared memory with 3-D TMA loads, kStages chunks ahead,
//     completing on one mbarrier per stage. When the layout does not meet
//     TMA's 16-byte rules the CTA fills the same tiles with plain loads;
//   - per chunk the CTA widens the B / C tiles to fp32 once for all of its
//     channels (double-buffered) and passes one barrier;
//   - steps are taken in groups of LPC: lane q of a channel computes dt =
//     softplus(delta + bias) for step q of the group and the LPC lanes trade
//     (dt, u) by warp shuffles; after the group's LPC recurrence steps the
//     lanes' partial readouts are reduce-scattered by shuffles so that lane q
//     holds the full y of step q, adds D u, applies the SiLU gate and stores
//     it. With LPC == 1 a thread does all of this for its own channel;
//   - bf16 inputs use the fast path: a scaled state s = A h, so that one step
//     is s <- s + (Abar - 1)(s + B u), and y = sum (C / A) s, all on packed
//     f32x2 FMUL/FFMA pairs of states, with Abar by MUFU ex2 and Abar - 1 =
//     ex2 - 1. Where dt |A| is small, ex2 - 1 loses the input term to
//     cancellation (relative error near 2^-23 / |dt A|). So every chunk runs
//     optimistically: each thread saves its state to shared memory, runs the
//     chunk with ex2 - 1 keeping the smallest dt it met, and compares that
//     with its channel's bound (dt |A| = 2^-14 for the channel's smallest
//     |A|). If a lane of the warp fell below, the warp restores its state and
//     runs the chunk again with Abar - 1 from a short series (expm1_acc),
//     overwriting the chunk's outputs; its inputs are still staged. The common
//     path pays one min per step group and four 16-byte stores per chunk, and its
//     unrolled step loop carries no branch. |A| is floored at 1e-20, where Abar and (Abar - 1) / A equal
//     their A -> 0 limits (1 and dt) in fp32 ("State Space Models and Mamba"
//     §2, the zero-order hold's limit). fp32 inputs use the precise path on
//     the unscaled state with expm1f, so that (Abar - 1) / A keeps full
//     relative accuracy.
//
// With CONV the kernel also runs the step in front of the scan in the Mamba
// block: u = SiLU(causal depthwise conv1d(x) + bias), width <= 4 ("Mamba"
// paper notes, Design 3; compassingai "Mamba" §3.3), from a u tile that TMA
// starts kConvHalo rows before the chunk (rows before t = 0 read as zero).
//
// With DISC = 1 the input matrix is the simplified Bbar = dt B of the "Mamba"
// paper notes' selective_ssm sketch (a follow-up option, not the method's ZOH):
// the state is kept unscaled and one step costs four FP32 lane-ops per state.
//
// Time segments (the split-L two-pass scheme): with nseg > 1 the aggregate
// pass (AGG = true) runs segments 0..nseg-2 from h = 0 and writes each
// segment's end state and sum of dt; the full pass then starts segment k from
// the composition of the aggregates 0..k-1 under the scan operator
// (a, b) o (a', b') = (a a', a' b + b'), where the decay of a whole segment is
// exp(A_n * sum dt) because A is constant in time ("State Space Models and
// Mamba" §4, parallel scan).
#pragma once

#include <type_traits>

#include "device_common.cuh"
#include "scan_args.h"

namespace mamba {

constexpr size_t scan_a128(size_t x) { return (x + 127) & ~size_t(127); }

// Steps of input before a chunk that the fused causal conv1d reads (width <= 4).
constexpr int kConvHalo = 3;

template <typename Tin, int NPL, int LPC, bool CONV = false>
struct ScanGeom {
  static constexpr int kCB = kScanThreads / LPC;  // channels per CTA
  static constexpr int kNP = NPL * LPC;           // padded state count
  static constexpr int kES = int(sizeof(Tin));
  static constexpr int kChunk = 16;               // steps per pipeline stage (a multiple of LPC)
  static constexpr int kStages = 3;               // TMA pipeline depth (chunks in flight)
  static constexpr int kURows = kChunk + (CONV ? kConvHalo : 0);  // rows of the u (or conv input) tile
  static constexpr size_t kUTile = scan_a128(size_t(kURows) * kCB * kES);
  static constexpr size_t kXTile = scan_a128(size_t(kChunk) * kCB * kES);
  static constexpr size_t kBCTile = scan_a128(size_t(kChunk) * kNP * kES);
  static constexpr size_t kStage = kUTile + 2 * kXTile + 2 * kBCTile;
  static constexpr size_t kBC32 = scan_a128(size_t(kChunk) * 2 * kNP * 4);  // [t][B | C][NP] fp32, x2 buffers
  static constexpr size_t kChan = scan_a128(size_t(kCB) * 2 * 4);           // bias, D per channel
  static constexpr size_t kSave = scan_a128(size_t(kScanThreads) * NPL * 4);  // each thread's state at a chunk start
  static constexpr size_t kBar = 128;
  static constexpr size_t kOffBC32 = kStages * kStage;
  static constexpr size_t kOffChan = kOffBC32 + 2 * kBC32;
  static constexpr size_t kOffSave = kOffChan + kChan;
  static constexpr size_t kOffBar = kOffSave + kSave;
  static constexpr size_t kSmem = kOffBar + kBar + 128;  // + alignment slack of the dynamic base
  static_assert(kChunk % LPC == 0, "a chunk holds whole step groups");
  static_assert(kSmem <= 227 * 1024, "scan variant exceeds the shared memory of one CTA");
  static_assert(NPL % 4 == 0, "states per thread come in groups of four (128-bit B / C loads)");
};

// One step of the fast path for NPL states held as NPL/2 packed pairs:
// s <- s + em1 (s + B u) with em1 = Abar - 1, Abar = 2^(dt * Ak), and (READ)
// the partial readout sum_j (C_j * Ik_j) s_j. ACC selects how em1 is formed:
// ex2 - 1 (false) or expm1_acc (true, exact to a few ulp at any dt A). Bt / Ct
// point at this thread's states.
template <int NPL, bool READ, bool ACC>
__device__ __forceinline__ float step_fast(float2 (&s)[NPL / 2], const float2 (&Ak)[NPL / 2],
                                           const float2 (&Ik)[NPL / 2], float dt, float u, const float* Bt,
                                           const float* Ct) {
  const float2 dd = make_float2(dt, dt);
  const float2 uu = make_float2(u, u);
  float2 yy[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};  // two chains of the readout sum
#pragma unroll
  for (int j = 0; j < NPL / 2; j += 2) {
    const float4 B4 = *reinterpret_cast<const float4*>(Bt + 2 * j);
    float4 C4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (READ) C4 = *reinterpret_cast<const float4*>(Ct + 2 * j);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 Bp = h == 0 ? make_float2(B4.x, B4.y) : make_float2(B4.z, B4.w);
      const float2 x = __fmul2_rn(dd, Ak[j + h]);
      const float2 ab = make_float2(hw_ex2(x.x), hw_ex2(x.y));
      float2 em1;
      if constexpr (ACC)
        em1 = make_float2(expm1_acc(x.x, ab.x), expm1_acc(x.y, ab.y));
      else
        em1 = __fadd2_rn(ab, make_float2(-1.0f, -1.0f));
      s[j + h] = __ffma2_rn(em1, __ffma2_rn(Bp, uu, s[j + h]), s[j + h]);
      if (READ) {
        const float2 Cp = h == 0 ? make_float2(C4.x, C4.y) : make_float2(C4.z, C4.w);
        yy[h] = __ffma2_rn(__fmul2_rn(Cp, Ik[j + h]), s[j + h], yy[h]);
      }
    }
  }
  return (yy[0].x + yy[1].x) + (yy[0].y + yy[1].y);
}

// One step of the precise path (unscaled state, expm1f): h <- h + (Abar - 1) h
// + (Abar - 1) / A * B u, readout sum_j C_j h_j. Ak holds A, Ik holds 1 / A.
template <int NPL, bool READ>
__device__ __forceinline__ float step_precise(float2 (&h)[NPL / 2], const float2 (&Ak)[NPL / 2],
                                              const float2 (&Ik)[NPL / 2], float dt, float u, const float* Bt,
                                              const float* Ct) {
  float y = 0.0f;
#pragma unroll
  for (int j = 0; j < NPL / 2; ++j) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float A = k == 0 ? Ak[j].x : Ak[j].y;
      const float I = k == 0 ? Ik[j].x : Ik[j].y;
      float& hv = k == 0 ? h[j].x : h[j].y;
      const float x = dt * A;
      const float e = expm1f(x);                     // Abar - 1
      const float coef = (x != 0.0f) ? e * I : dt;   // (Abar - 1) / A, limit dt
      hv = fmaf(coef * Bt[2 * j + k], u, fmaf(e, hv, hv));
      if (READ) y = fmaf(Ct[2 * j + k], hv, y);
    }
  }
  return y;
}

// Simplified discretisation (Bbar = dt B, the "Mamba" paper notes' selective_ssm
// sketch), fast path on the unscaled state: h <- Abar h + (dt u) B with Abar =
// 2^(dt * Ak), readout sum_j C_j h_j. Four FP32 lane-ops per state instead of six.
template <int NPL, bool READ>
__device__ __forceinline__ float step_fast_simple(float2 (&h)[NPL / 2], const float2 (&Ak)[NPL / 2], float dt,
                                                  float u, const float* Bt, const float* Ct) {
  const float2 dd = make_float2(dt, dt);
  const float du = dt * u;
  const float2 dud = make_float2(du, du);
  float2 yy[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int j = 0; j < NPL / 2; j += 2) {
    const float4 B4 = *reinterpret_cast<const float4*>(Bt + 2 * j);
    float4 C4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (READ) C4 = *reinterpret_cast<const float4*>(Ct + 2 * j);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 Bp = k == 0 ? make_float2(B4.x, B4.y) : make_float2(B4.z, B4.w);
      const float2 x = __fmul2_rn(dd, Ak[j + k]);
      const float2 ab = make_float2(hw_ex2(x.x), hw_ex2(x.y));
      h[j + k] = __ffma2_rn(ab, h[j + k], __fmul2_rn(Bp, dud));
      if (READ) {
        const float2 Cp = k == 0 ? make_float2(C4.x, C4.y) : make_float2(C4.z, C4.w);
        yy[k] = __ffma2_rn(Cp, h[j + k], yy[k]);
      }
    }
  }
  return (yy[0].x + yy[1].x) + (yy[0].y + yy[1].y);
}

// Simplified discretisation, precise path: h <- exp(dt A) h + dt B u.
template <int NPL, bool READ>
__device__ __forceinline__ float step_precise_simple(float2 (&h)[NPL / 2], const float2 (&Ak)[NPL / 2], float dt,
                                                     float u, const float* Bt, const float* Ct) {
  float y = 0.0f;
  const float du = dt * u;
#pragma unroll
  for (int j = 0; j < NPL / 2; ++j) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float A = k == 0 ? Ak[j].x : Ak[j].y;
      float& hv = k == 0 ? h[j].x : h[j].y;
      hv = fmaf(expf(dt * A), hv, du * Bt[2 * j + k]);
      if (READ) y = fmaf(Ct[2 * j + k], hv, y);
    }
  }
  return y;
}

// Sum over the LPC lanes of a channel of v[0..LPC), scattered so that lane q
// returns the total of entry q: recursive halving over xor partners, one
// round per bit of q from the highest (M = LPC / 2) down to 1. Written as a
// compile-time recursion so that every index into v is static.
template <int M, int LPC>
__device__ __forceinline__ void reduce_scatter_round(float (&v)[LPC], int q) {
  if constexpr (M >= 1) {
    const bool hi = (q & M) != 0;
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const float send = hi ? v[i] : v[i + M];
      const float keep = hi ? v[i + M] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
    }
    reduce_scatter_round<M / 2, LPC>(v, q);
  }
}

template <int LPC>
__device__ __forceinline__ float reduce_scatter(float (&v)[LPC], int q) {
  reduce_scatter_round<LPC / 2, LPC>(v, q);
  return v[0];
}

// CTAs per SM each variant's register budget is sized for: 4 (<= 128
// registers per thread) for every state split. The scans these plans serve are
// latency-bound at a few CTAs per SM, and the registers let the compiler move a
// step group's softplus, loads and exponentials ahead of the state chain. On
// B300 the 4-state variant on the 130M-shaped layer (2.6 CTAs per SM) went from
// 277 us at 8 CTAs per SM (64 registers) to 239 us; 5 and 6 gave 251 and 265 us,
// and a layer with 7 CTAs per SM ran the same with either budget.
template <int NPL>
struct ScanMinBlocks {
  static constexpr int value = 4;
};

// DISC: 0 = zero-order hold (the method), 1 = simplified Bbar = dt B.
// CONV: the u argument holds the conv input x; u = SiLU(causal conv1d(x)) is
// computed on the fly (conv_w, conv_b, conv_width of ScanArgs).
template <typename Tin, int NPL, int LPC, bool AGG, int DISC, bool CONV>
__global__ void __launch_bounds__(kScanThreads, ScanMinBlocks<NPL>::value)
    scan_kernel(const ScanArgs a, const __grid_constant__ ScanMaps maps) {
  using G = ScanGeom<Tin, NPL, LPC, CONV>;
  using E = Elem<Tin>;
  constexpr bool PRECISE = std::is_same<Tin, float>::value;
  constexpr bool SCALED = !PRECISE && DISC == 0;  // fast ZOH path keeps s = A h
  constexpr int CB = G::kCB, NP = G::kNP, CH = G::kChunk, NS = G::kStages;
  constexpr int NH = NPL / 2;

  extern __shared__ unsigned char smem_dyn[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  float* chan_bias = reinterpret_cast<float*>(smem + G::kOffChan);
  float* chan_D = chan_bias + CB;
  float4* save = reinterpret_cast<float4*>(smem + G::kOffSave);  // [NPL / 4][threads]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + G::kOffBar);

  // Stage s: u tile (kURows rows; with CONV its first kConvHalo rows are the
  // inputs before the chunk), delta and z tiles, B and C tiles.
  auto xu = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage); };
  auto xd = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kUTile); };
  auto xz = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kUTile + G::kXTile); };
  auto braw = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kUTile + 2 * G::kXTile); };
  auto craw = [&](int s) {
    return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kUTile + 2 * G::kXTile + G::kBCTile);
  };
  constexpr int UH = CONV ? kConvHalo : 0;  // halo rows at the top of the u tile
  auto bc32 = [&](int k) { return reinterpret_cast<float*>(smem + G::kOffBC32 + (k & 1) * G::kBC32); };

  const int tid = threadIdx.x;
  const int c = tid / LPC, q = tid % LPC;
  const int Dm = a.dim, N = a.dstate, L = a.seqlen;
  const int d0 = blockIdx.x * CB;
  const int d = d0 + c;
  const bool dvalid = d < Dm;
  const int b = blockIdx.y;
  const int seg = blockIdx.z;
  const int t_begin = seg * a.seg_len;
  const int t_end = min(L, t_begin + a.seg_len);
  const int nchunks = (t_end - t_begin + CH - 1) / CH;
  const bool has_z = !AGG && a.z != nullptr;
  const bool use_tma = a.tma_x || a.tma_bc;
  const Tin* gu = static_cast<const Tin*>(a.u);
  const Tin* gdl = static_cast<const Tin*>(a.delta);
  const Tin* gz = static_cast<const Tin*>(a.z);
  const Tin* gB = static_cast<const Tin*>(a.B);
  const Tin* gC = static_cast<const Tin*>(a.C);
  // The next kernel in the stream may start its prologue while this grid runs
  // (it waits before it reads what this grid writes).
  griddep_launch();

  // Per-channel constants of this CTA.
  for (int i = tid; i < CB; i += kScanThreads) {
    const int dd = d0 + i;
    chan_bias[i] = (a.delta_bias && dd < Dm) ? a.delta_bias[dd] : 0.0f;
    chan_D[i] = (a.D && dd < Dm) ? a.D[dd] : 0.0f;
  }

  // Chunk staging by TMA (thread 0 only).
  auto issue = [&](int k) {
    const int s = k % NS;
    const int t0 = t_begin + k * CH;
    uint32_t bytes = 0;
    if (a.tma_x) bytes += uint32_t(((has_z ? 2 : 1) * CH + G::kURows) * CB * sizeof(Tin));
    if (a.tma_bc) bytes += 2u * uint32_t(CH * N * sizeof(Tin));
    mbar_arrive_expect_tx(&mbar[s], bytes);
    if (a.tma_x) {
      tma_load_3d(xu(s), &maps.u, d0, t0 - UH, b, &mbar[s]);  // rows before 0 read as zero
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
    if (a.tma_x) {
      prefetch_tensormap(&maps.u);
      prefetch_tensormap(&maps.delta);
      if (has_z) prefetch_tensormap(&maps.z);
    }
    if (a.tma_bc) {
      prefetch_tensormap(&maps.B);
      prefetch_tensormap(&maps.C);
    }
  }
  __syncthreads();
  int issued = 0;  // chunks handed to TMA so far (thread 0)
  if (use_tma && tid == 0)
    for (; issued < min(NS, nchunks); ++issued) issue(issued);

  // Per-thread constants for my NPL states:
  //  fast:    Ak = A * log2(e) (exponent for ex2), Ik = 1 / A;
  //  precise: Ak = A,                              Ik = 1 / A.
  // A = -exp(A_log) with |A| >= kMinAbsA.
  float2 Ak[NH], Ik[NH], st[NH];
  float Av[NPL], hin[NPL];
  float minA = 3.0e38f;  // smallest |A| of my real states
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int n = q * NPL + j;
    const bool real = n < N;
    float A = -1.0f;
    if (dvalid && real) A = -expf(a.A_log[(size_t)d * N + n]);
    A = fminf(A, -kMinAbsA);
    if (real) minA = fminf(minA, -A);
    Av[j] = A;
    const float ak = real ? (PRECISE ? A : A * kLog2e) : 0.0f;
    const float ik = real ? 1.0f / A : 0.0f;
    hin[j] = (!AGG && real && dvalid && a.h0) ? a.h0[((size_t)b * Dm + d) * N + n] : 0.0f;
    if (j % 2 == 0) {
      Ak[j / 2].x = ak;
      Ik[j / 2].x = ik;
    } else {
      Ak[j / 2].y = ak;
      Ik[j / 2].y = ik;
    }
  }
  // Initial state of my segment: h0 (or 0) composed with the aggregates of
  // the earlier segments, oldest first. The segments are the outer loop and
  // my NPL aggregate values are read as 16-byte vectors where N allows, so
  // that the loads of several segments are in flight at once (they do not
  // depend on the state being composed).
  // A full pass that follows the aggregate pass may have started before that
  // pass ended: it has staged its first chunks of inputs (which the aggregate
  // pass does not write) and now waits for the aggregates.
  if (!AGG && a.after_agg && seg > 0) griddep_wait();
  if (!AGG && dvalid && seg > 0) {
    const bool vec = (N % 4) == 0 && (q + 1) * NPL <= N;  // all my states real: the vectors stay in the row
#pragma unroll 4
    for (int k = 0; k < seg; ++k) {
      const size_t row = (size_t)b * (a.nseg - 1) + k;
      const float ds = a.agg_dsum[row * Dm + d];
      const float* ah = a.agg_h + (row * Dm + d) * N + q * NPL;
      float e[NPL];
#pragma unroll
      for (int j = 0; j < NPL; j += 4) {
        if (vec) {
          const float4 v = *reinterpret_cast<const float4*>(ah + j);
          e[j] = v.x; e[j + 1] = v.y; e[j + 2] = v.z; e[j + 3] = v.w;
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) e[j + i] = (q * NPL + j + i < N) ? ah[j + i] : 0.0f;
        }
      }
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const float ak = (j % 2 == 0) ? Ak[j / 2].x : Ak[j / 2].y;
        const float decay = PRECISE ? expf(Av[j] * ds) : hw_ex2(ak * ds);
        hin[j] = fmaf(decay, hin[j], e[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const float sv = SCALED ? hin[j] * Av[j] : hin[j];
    if (j % 2 == 0) st[j / 2].x = sv;
    else st[j / 2].y = sv;
  }
  const float bias = chan_bias[c];
  const float Dd = chan_D[c];
  // dt below which a step of my channel needs the accurate Abar - 1
  float thr = 0.0f;
  if constexpr (SCALED) {
#pragma unroll
    for (int o = 1; o < LPC; o <<= 1) minA = fminf(minA, __shfl_xor_sync(0xffffffffu, minA, o));
    thr = kFastMinDtA / minA;
  }
  // Conv taps aligned to the u tile: tap j multiplies row tm + j (input step
  // t - kConvHalo + j), so a width-W kernel fills taps kConvHalo + 1 - W .. kConvHalo.
  float cw[kConvHalo + 1] = {0.0f, 0.0f, 0.0f, 0.0f};
  float cb = 0.0f;
  if constexpr (CONV) {
    if (dvalid) {
      const int W = a.conv_width;
#pragma unroll
      for (int j = 0; j <= kConvHalo; ++j) {
        const int k = j - (kConvHalo + 1 - W);
        cw[j] = (k >= 0) ? a.conv_w[(size_t)d * W + k] : 0.0f;
      }
      cb = a.conv_b ? a.conv_b[d] : 0.0f;
    }
  }

  float dsum = 0.0f;    // AGG: sum of dt over the segment (fast path)
  double dsum_d = 0.0;  // AGG: the same in fp64 (precise path)

  // The steps of one staged chunk (see the loop below).
  // Returns (fast path) whether a lane of the warp met a step with dt < thr
  // (steps past the end count too: a ragged last chunk may be rerun for nothing).
  auto run_chunk = [&]<bool HZ, bool ACC>(int s, int kc, int t0, int tv) -> bool {
    [[maybe_unused]] float dtmin = 3.0e38f;
    const Tin* su = xu(s) + c;
    const Tin* sd = xd(s) + c;
    const Tin* sz = xz(s) + c;
    const float* bcq = bc32(kc) + q * NPL;
    Tin* gout = static_cast<Tin*>(a.out) + ((size_t)b * L + t0 + q) * Dm + d;
    (void)gout;
    // dt and u of step q of the first group, computed by this lane
    auto lane_dtu = [&](int tm, float& dtv, float& uv) {
      float um;
      if constexpr (CONV) {
        float acc = cb;
#pragma unroll
        for (int j = 0; j <= kConvHalo; ++j) acc = fmaf(cw[j], E::load(su + (tm + j) * CB), acc);
        um = PRECISE ? silu_precise(acc) : silu_fast(acc);
      } else {
        um = E::load(su + tm * CB);
      }
      const float xm = E::load(sd + tm * CB) + bias;
      const float dt = PRECISE ? softplus_precise(xm) : softplus_fast(xm);
      const bool live = tm < tv;
      dtv = live ? dt : 0.0f;
      uv = live ? um : 0.0f;
      if constexpr (SCALED && !ACC) dtmin = fminf(dtmin, dt);
    };
    float dt_nx, u_nx;
    lane_dtu(q, dt_nx, u_nx);
    [[maybe_unused]] float y_pv = 0.0f, u_pv = 0.0f, z_pv = 0.0f;  // previous group's readout, pending its epilogue
#pragma unroll 4
    for (int tg = 0; tg < CH; tg += LPC) {
      const float dt_cu = dt_nx, u_cu = u_nx;
      float z_cu = 0.0f;
      if (!AGG && HZ) z_cu = E::load(sz + (tg + q) * CB);
      if (tg + LPC < CH) lane_dtu(tg + LPC + q, dt_nx, u_nx);
      float yp[LPC];
#pragma unroll
      for (int j = 0; j < LPC; ++j) {
        const int src = (tid & 31) - q + j;
        const float dt = LPC == 1 ? dt_cu : __shfl_sync(0xffffffffu, dt_cu, src);
        const float u = LPC == 1 ? u_cu : __shfl_sync(0xffffffffu, u_cu, src);
        const float* Bt = bcq + (tg + j) * 2 * NP;
        if constexpr (DISC == 1 && PRECISE)
          yp[j] = step_precise_simple<NPL, !AGG>(st, Ak, dt, u, Bt, Bt + NP);
        else if constexpr (DISC == 1)
          yp[j] = step_fast_simple<NPL, !AGG>(st, Ak, dt, u, Bt, Bt + NP);
        else if constexpr (PRECISE)
          yp[j] = step_precise<NPL, !AGG>(st, Ak, Ik, dt, u, Bt, Bt + NP);
        else
          yp[j] = step_fast<NPL, !AGG, ACC>(st, Ak, Ik, dt, u, Bt, Bt + NP);
        if constexpr (AGG) {
          if (PRECISE) dsum_d += dt; else dsum += dt;
        }
      }
      if constexpr (!AGG) {
        // epilogue of the previous group: D skip, gate, store
        if (tg > 0) {
          float y = fmaf(Dd, u_pv, y_pv);
          if (HZ) y *= PRECISE ? silu_precise(z_pv) : silu_fast(z_pv);
          if (dvalid && tg - LPC + q < tv) E::store(gout + (size_t)(tg - LPC) * Dm, y);
        }
        y_pv = reduce_scatter<LPC>(yp, q);  // full readout of step tg + q
        u_pv = u_cu;
        z_pv = z_cu;
      }
    }
    if constexpr (!AGG) {
      float y = fmaf(Dd, u_pv, y_pv);
      if (HZ) y *= PRECISE ? silu_precise(z_pv) : silu_fast(z_pv);
      if (dvalid && CH - LPC + q < tv) E::store(gout + (size_t)(CH - LPC) * Dm, y);
    }
    if constexpr (SCALED && !ACC) return __any_sync(0xffffffffu, dtmin < thr);
    return false;
  };

  for (int k = 0; k < nchunks; ++k) {
    const int s = k % NS;
    const int t0 = t_begin + k * CH;
    const int tv = min(CH, t_end - t0);

    if (use_tma) {
      const bool ok = mbar_wait_bounded(&mbar[s], (k / NS) & 1, a.wait_ns);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          record_status(a.status, kStatusTimeout);
          // Let copies already in flight land before the CTA's shared memory goes away.
          for (int kk = k; kk < issued; ++kk) mbar_wait_bounded(&mbar[kk % NS], (kk / NS) & 1);
        }
        return;
      }
    }
    // Plain loads into the tiles where TMA cannot be used (zero outside the tensor).
    if (!a.tma_x) {
      for (int i = tid; i < G::kURows * CB; i += kScanThreads) {
        const int t = i / CB, cc = i % CB;
        const int gt = t0 - UH + t, gd = d0 + cc;
        const bool in = gt >= 0 && gt < L && gd < Dm;
        xu(s)[i] = in ? gu[((size_t)b * L + gt) * Dm + gd] : Tin(0.0f);
      }
      for (int i = tid; i < CH * CB; i += kScanThreads) {
        const int t = i / CB, cc = i % CB;
        const int gt = t0 + t, gd = d0 + cc;
        const bool in = gt < L && gd < Dm;
        const size_t off = ((size_t)b * L + gt) * Dm + gd;
        xd(s)[i] = in ? gdl[off] : Tin(0.0f);
        if (has_z) xz(s)[i] = in ? gz[off] : Tin(0.0f);
      }
    }
    // B / C rows widened to fp32 once for every channel of the CTA (zero beyond N).
    float* bck = bc32(k);
    for (int i = tid; i < CH * NP; i += kScanThreads) {
      const int t = i / NP, n = i % NP;
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
      bck[t * 2 * NP + n] = bv;
      bck[t * 2 * NP + NP + n] = cv;
    }
    __syncthreads();  // chunk k staged; every thread is past chunk k-1
    if (use_tma && tid == 0 && k >= 1 && issued < nchunks) {
      fence_proxy_async_smem();  // chunk k-1's stage was read through the generic proxy
      issue(issued);
      ++issued;
    }

    // ---- the recurrence over chunk k, in groups of LPC steps. Every chunk
    // runs all CH steps: steps at or past tv (the end of the sequence or of
    // the segment) get dt = 0 and u = 0, which leaves the state exactly as it
    // is (Abar = 1, no input), and store nothing. The loop is branch-free and
    // fully unrolled so that the compiler can overlap a group's recurrence
    // with the next group's softplus and the previous group's epilogue.
    if constexpr (SCALED) {
      // optimistic fast pass; the warp reruns the chunk accurately if it met a small dt |A|
#pragma unroll
      for (int j = 0; j < NH; j += 2) save[(j / 2) * kScanThreads + tid] = make_float4(st[j].x, st[j].y, st[j + 1].x, st[j + 1].y);
      const float dsum0 = dsum;
      const bool redo = has_z ? run_chunk.template operator()<true, false>(s, k, t0, tv)
                              : run_chunk.template operator()<false, false>(s, k, t0, tv);
      if (redo) {
#pragma unroll
        for (int j = 0; j < NH; j += 2) {
          const float4 v = save[(j / 2) * kScanThreads + tid];
          st[j] = make_float2(v.x, v.y);
          st[j + 1] = make_float2(v.z, v.w);
        }
        dsum = dsum0;
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

  if (!dvalid) return;
  if constexpr (AGG) {
    const size_t row = (size_t)b * (a.nseg - 1) + seg;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int n = q * NPL + j;
      const float sv = (j % 2 == 0) ? st[j / 2].x : st[j / 2].y;
      const float ik = (j % 2 == 0) ? Ik[j / 2].x : Ik[j / 2].y;
      if (n < N) a.agg_h[(row * Dm + d) * N + n] = SCALED ? sv * ik : sv;
    }
    if (q == 0) a.agg_dsum[row * Dm + d] = PRECISE ? float(dsum_d) : dsum;
  } else {
    if (a.last_state && seg == a.nseg - 1) {
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int n = q * NPL + j;
        const float sv = (j % 2 == 0) ? st[j / 2].x : st[j / 2].y;
        const float ik = (j % 2 == 0) ? Ik[j / 2].x : Ik[j / 2].y;
        if (n < N) a.last_state[((size_t)b * Dm + d) * N + n] = SCALED ? sv * ik : sv;
      }
    }
  }
}

// Launch one (dtype, NPL, LPC, mode) instantiation.
template <typename Tin, int DISC, bool CONV, int NPL, int LPC>
cudaError_t launch_scan_variant(ScanMode mode, const ScanArgs& a, const ScanMaps& maps, dim3 grid,
                                cudaStream_t stream) {
  using G = ScanGeom<Tin, NPL, LPC, CONV>;
  auto kfull = scan_kernel<Tin, NPL, LPC, false, DISC, CONV>;
  auto kagg = scan_kernel<Tin, NPL, LPC, true, DISC, CONV>;
  static bool configured = false;  // per instantiation; benign race (idempotent)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kfull, cudaFuncAttributeMaxDynamicSharedMemorySize, int(G::kSmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, int(G::kSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (mode == ScanMode::kFull && a.after_agg) return launch_pdl(kfull, grid, dim3(kScanThreads), G::kSmem, stream, a, maps);
  if (mode == ScanMode::kFull)
    kfull<<<grid, kScanThreads, G::kSmem, stream>>>(a, maps);
  else
    kagg<<<grid, kScanThreads, G::kSmem, stream>>>(a, maps);
  return cudaGetLastError();
}

template <typename Tin, int NPL, int LPC>
void describe_variant(ScanVariant* v) {
  using G = ScanGeom<Tin, NPL, LPC>;
  v->npl = NPL;
  v->lpc = LPC;
  v->cb = G::kCB;
  v->chunk = G::kChunk;
  v->smem_bytes = G::kSmem;
}

// The (NPL, LPC) pairs that exist: N <= NPL * LPC <= 256, NPL in {4, 8, 16}.
#define MAMBA_SCAN_VARIANTS(X) \
  X(4, 1)                      \
  X(8, 1)                      \
  X(16, 1)                     \
  X(4, 2)                      \
  X(8, 2)                      \
  X(16, 2)                     \
  X(4, 4)                      \
  X(8, 4)                      \
  X(16, 4)                     \
  X(8, 8)                      \
  X(16, 8)                     \
  X(16, 16)

template <typename Tin, int DISC, bool CONV = false>
cudaError_t launch_scan_typed(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps, dim3 grid,
                              cudaStream_t stream) {
#define MAMBA_CASE(P, Q) \
  if (npl == P && lpc == Q) return launch_scan_variant<Tin, DISC, CONV, P, Q>(mode, a, maps, grid, stream);
  MAMBA_SCAN_VARIANTS(MAMBA_CASE)
#undef MAMBA_CASE
  return cudaErrorInvalidValue;
}

template <typename Tin>
bool scan_variant_typed(int npl, int lpc, ScanVariant* v) {
#define MAMBA_CASE(P, Q)                  \
  if (npl == P && lpc == Q) {             \
    describe_variant<Tin, P, Q>(v);       \
    return true;                          \
  }
  MAMBA_SCAN_VARIANTS(MAMBA_CASE)
#undef MAMBA_CASE
  return false;
}

}  // namespace mamba
