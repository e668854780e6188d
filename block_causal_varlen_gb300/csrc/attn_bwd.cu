// Backward of block-causal varlen chunked attention on sm_103a, head dim 64 and
// 128 (head dim 256 has its own kernel in attn_bwd256.cu).
//
// What it computes, for the loss sum(O * dO) (the analytic gradient of the
// forward of the NeMo Automodel page "block-diagonal varlen CP for packed
// sequences", with the fused K/V all-gather whose backward is a
// reduce-scatter SUM, Design overview exchange.py):
//   P_ij = exp(scale q_i.k_j - LSE_i) on the block-causal mask, else 0
//   dV_j = sum_i P_ij dO_i          dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i),     D_i = dO_i . O_i
//   dQ_i = scale sum_j dS_ij k_j    dK_j = scale sum_i dS_ij q_i
// dK/dV of a K/V head sum over the query heads of its GQA group and, for a
// shared (all-gathered) K/V buffer, over every chunk of the sequence: that sum
// is the reduce-scatter SUM done in place.
//
// Design (one persistent CTA per SM, 16 warps, each claiming its next work unit
// from a per-launch counter when it is ready for it). A work unit is one 128-row
// K/V tile of one K/V head; K and V stay in shared memory while the CTA walks
// every (query tile, query head of the group) step that attends to the tile.
//   warp 0       TMA producer: K/V once per unit; per step a Q tile (2-stage
//                ring, with the step's LSE / D / document-start rows) and a dO
//                tile.
//   warp 1       TMEM allocation; one thread issues the five tcgen05.mma per
//                step: S^T = K Q^T, dP^T = V dO^T (TMEM), dV += P^T dO (P^T read
//                from TMEM), dK += dS^T Q, dQ = dS K (dS^T from shared memory).
//   warps 4-11   P^T and dS^T for the tile's 128 keys (lane = key row), two
//                warps per lane quarter, one per 64-query half.
//   warps 12-15  read dQ out of TMEM and add it into global memory with TMA
//                reduce-adds (128 x 16 fp32 boxes staged through two shared
//                memory buffers); at the end of a unit write dK (x scale) and dV.
// TMEM columns: S^T/P^T [0,128), dP^T/dQ [128,256), dV, dK after that.
// The DROP instantiation regenerates the forward's dropout keep mask
// (Philox4x32-10 from the plan's seed): dV reads the dropped, rescaled P^T and
// dS = P (keep dP / (1 - p) - D) uses the undropped P.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "bwd_aux.h"
#include "bwd_kernel.cuh"
#include "host_util.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace bd {
using namespace dev;

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;          // two stages
  static constexpr int kOffDO = 4 * kTileBytes;
  static constexpr int kOffDS = 5 * kTileBytes;         // dS^T, 128 keys x 128 queries bf16
  static constexpr int kOffStat = kOffDS + 32768;       // per stage: lse2[128], D[128]
  static constexpr int kStatBytes = 2 * 512;
  // dQ staging: two buffers of one 128 rows x 32 columns fp32 reduce box (16 KB,
  // 128-byte swizzle): a TMA reduce-add costs ~425 cycles per box up to 8 KB and
  // ~712 for 16 KB, so 16 KB boxes move dQ ~20% faster than 8 KB ones
  static constexpr int kOffStage = kOffStat + 2 * kStatBytes;
  static constexpr int kStageBytes = 128 * 32 * 4;
  static constexpr int kOffBar = kOffStage + 2 * kStageBytes;
  // no alignment slack: the dynamic shared memory base must be 1024-byte aligned
  // (checked at kernel entry; the kernel records a failure and does nothing if not)
  static constexpr int kSmem = kOffBar + 256;
  static_assert(kSmem <= 232448, "shared memory over the per-CTA limit");
  static constexpr int kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr int kThreads = 512;
  // register split after setmaxnreg: producer/MMA, P/dS warpgroups, dQ warpgroup
  static constexpr int kRegsCtl = 96, kRegsCompute = 120, kRegsDq = 176;
  static constexpr int kRegsNeeded = 128 * kRegsCtl + 256 * kRegsCompute + 128 * kRegsDq;
  static constexpr int kRegsLaunch = 128;  // 65536 / 512 threads: what ptxas assigns at launch
  static_assert(kRegsNeeded <= kRegsLaunch * kThreads, "register split exceeds the launch's registers");
};

enum : int {
  C_KVFULL = 0, C_KVEMPTY, C_QFULL0, C_QFULL1, C_QEMPTY0, C_QEMPTY1, C_DOFULL, C_DOEMPTY, C_SFULL, C_DPFULL,
  C_PREADY, C_DSREADY, C_DQFULL, C_DQEMPTY, C_ACCDONE, C_DVFREE, C_DKFREE, C_DRAIN, C_UFULL,
  C_UEMPTY = C_UFULL + kUnitSlots, C_COUNT = C_UEMPTY + kUnitSlots
};
// warps that read each claimed unit from the ring: MMA thread, 8 P/dS warps, 4 dQ warps
constexpr uint32_t kUnitConsumers = 1 + 8 + 4;
static_assert(8 * C_COUNT + 16 + 4 * kUnitSlots <= 256, "barriers, TMEM slot, abort flag and unit ring overflow their region");

template <int D, bool DROP>
__global__ void __launch_bounds__(512, 1)
    bd_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, const BwdArgs a) {
  using Cfg = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  // the 128-byte-swizzled operand tiles need 1024-byte alignment and the layout
  // leaves no slack to round up: refuse (and record why) rather than overrun
  if (sbase & 1023u) {
    if (threadIdx.x == 0) {
      atomicExch(const_cast<int32_t*>(a.plan) + H_STATUS, DEV_SMEM_ALIGN);
      atomicExch(const_cast<int32_t*>(a.plan) + H_STATUS_DETAIL, 2);
    }
    return;
  }
  const uint32_t sK = sbase + Cfg::kOffK, sV = sbase + Cfg::kOffV, sQ = sbase + Cfg::kOffQ;
  const uint32_t sDO = sbase + Cfg::kOffDO, sDS = sbase + Cfg::kOffDS, sStage = sbase + Cfg::kOffStage;
  const uint32_t bars = sbase + Cfg::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffBar + 8 * C_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffBar + 8 * C_COUNT + 8);
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Cfg::kOffBar + 8 * C_COUNT + 16);
  int* claim = a.counters;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t* plan = a.plan;
  const int32_t* work = plan + a.work_off;
  const int32_t* items = plan + plan[H_OFF_ITEMS];

  if (threadIdx.x == 0) {
    for (int i = 0; i < C_COUNT; ++i) {
      const uint32_t n = (i == C_PREADY || i == C_DSREADY)       ? 256u
                         : (i == C_DQEMPTY || i == C_DVFREE || i == C_DKFREE) ? 128u
                         : (i >= C_UEMPTY && i < C_UEMPTY + kUnitSlots) ? kUnitConsumers
                                                                       : 1u;
      mbar_init(bar(i), n);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // registers move from warpgroup 0 (producer, MMA) to the compute warpgroups at
  // the top of each warpgroup's branch
  if (warp < 4) {
   regs_set<Cfg::kRegsCtl, Cfg::kRegsLaunch>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t u = 0, sc = 0, q_iss = 0, do_iss = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        const int w = unit_publish(bar(C_UFULL), bar(C_UEMPTY), unit_ring, claim, a.n_work, uk, abort_flag);
        if (w == -2) ok = false;
        if (w < 0) break;
        const int32_t* W = work + w * kBwdWords;
        if (W[W_NQ] == 0) continue;
        const int g = W[W_G], kb = W[W_BUF] / a.Ck, kc = W[W_BUF] % a.Ck;
        if (!(ok = mbar_wait(bar(C_KVEMPTY), (u & 1) ^ 1, abort_flag))) break;
        mbar_expect_tx(bar(C_KVFULL), 2 * Cfg::kTileBytes);
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_5d(sK + hf * 16384, &tm_k, bar(C_KVFULL), hf * 64, g, W[W_LROW], kc, kb);
          tma_load_5d(sV + hf * 16384, &tm_v, bar(C_KVFULL), hf * 64, g, W[W_LROW], kc, kb);
        }
        ++u;
        const StepRange<128> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
        // Q / dO / row statistics of a step are loaded once its stage is free (the
        // stage's previous Q is read by the last MMA of the step before); an L2
        // prefetch of the next step's tiles measured no gain
        struct Step { int it, t, h, b, c; };
        Step prev{};
        bool have_prev = false;
        auto load_step = [&](const Step& x) {
          const int qs = sc & 1;
          if (!(ok = mbar_wait(bar(C_QEMPTY0 + qs), ((sc >> 1) & 1) ^ 1, abort_flag))) return;
          mbar_expect_tx(bar(C_QFULL0 + qs), Cfg::kTileBytes + Cfg::kStatBytes);
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_5d(sQ + qs * Cfg::kTileBytes + hf * 16384, &tm_q, bar(C_QFULL0 + qs), hf * 64, x.h, x.t * 128,
                        x.c, x.b);
          const uint32_t st = sbase + Cfg::kOffStat + qs * Cfg::kStatBytes;
          const int64_t srow = (int64_t(x.it) * a.H + x.h) * a.Lpad + x.t * 128;
          bulk_load(st, a.lse2 + srow, 512, bar(C_QFULL0 + qs));
          bulk_load(st + 512, a.dstat + srow, 512, bar(C_QFULL0 + qs));
          ++q_iss;
          if (!(ok = mbar_wait(bar(C_DOEMPTY), (sc & 1) ^ 1, abort_flag))) return;
          mbar_expect_tx(bar(C_DOFULL), Cfg::kTileBytes);
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_5d(sDO + hf * 16384, &tm_do, bar(C_DOFULL), hf * 64, x.h, x.t * 128, x.c, x.b);
          ++do_iss;
          ++sc;
        };
        for (int it = R.it_lo; it < R.it_hi && ok; ++it) {
          int t0, t1, r0;
          if (!R.tiles(it, t0, t1, r0)) continue;
          const int32_t* I = items + it * kItemWords;
          const int b = I[I_B], c = I[I_C];
          for (int t = t0; t <= t1 && ok; ++t)
            for (int hh = 0; hh < a.G && ok; ++hh) {
              const Step x{it, t, g * a.G + hh, b, c};
              if (have_prev) load_step(prev);
              prev = x;
              have_prev = true;
            }
        }
        if (have_prev && ok) load_step(prev);
      }
      if (!ok) {
        // wait for copies already issued before the shared memory goes away
        if (u > 0) mbar_wait_drain(bar(C_KVFULL), (u - 1) & 1);
        for (uint32_t x = (q_iss > 2 ? q_iss - 2 : 0); x < q_iss; ++x)
          mbar_wait_drain(bar(C_QFULL0 + (x & 1)), (x >> 1) & 1);
        if (do_iss > 0) mbar_wait_drain(bar(C_DOFULL), (do_iss - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idKM = idesc_bf16(128, D, false, true);   // A K-major, B MN-major
      constexpr uint32_t idMM = idesc_bf16(128, D, true, true);    // both MN-major
      // base descriptors of every operand tile are built once; a K step only
      // advances the start-address field (16-byte units) with a 64-bit add
      const uint32_t dK_k = sdesc_lo(sK, 16), dV_k = sdesc_lo(sV, 16), dK_mn = sdesc_lo(sK, 16384);
      const uint32_t dDO_k = sdesc_lo(sDO, 16), dDO_mn = sdesc_lo(sDO, 16384);
      const uint32_t dDS_k = sdesc_lo(sDS, 16), dDS_mn = sdesc_lo(sDS, 16384);
      auto dQ_k = [&](int qs) { return sdesc_lo(sQ + qs * Cfg::kTileBytes, 16); };
      auto dQ_mn = [&](int qs) { return sdesc_lo(sQ + qs * Cfg::kTileBytes, 16384); };
      auto kstep = [](int kk) { return uint32_t(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
      auto mnstep = [](int kk) { return uint32_t((kk * 2048) >> 4); };
      uint32_t u = 0, sc = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        const int w = unit_take(bar(C_UFULL), bar(C_UEMPTY), unit_ring, uk, abort_flag, true);
        if (w == -2) ok = false;
        if (w < 0) break;
        const int32_t* W = work + w * kBwdWords;
        const int nsteps = W[W_NQ];
        if (nsteps == 0) continue;
        if (!(ok = mbar_wait(bar(C_KVFULL), u & 1, abort_flag))) break;
        auto issue_s = [&](uint32_t step) {  // S^T = K Q^T for the Q tile of `step`
          const uint32_t qd = dQ_k(step & 1);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) mma_ss_lo(tmem, dK_k + kstep(kk), qd + kstep(kk), idSS, kk > 0);
          tc_commit(bar(C_SFULL));
        };
        if (!(ok = mbar_wait(bar(C_QFULL0 + (sc & 1)), (sc >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        issue_s(sc);
        for (int s = 0; s < nsteps && ok; ++s, ++sc) {
          const int qs = sc & 1;
          BD_TRACE_EVENT(0, int(sc));  // MMA: step start (waits dO, dQ drained)
          if (!(ok = mbar_wait(bar(C_DOFULL), sc & 1, abort_flag))) break;
          BD_TRACE_EVENT(1, int(sc));
          if (!(ok = mbar_wait(bar(C_DQEMPTY), (sc & 1) ^ 1, abort_flag))) break;
          BD_TRACE_EVENT(2, int(sc));  // MMA: dP^T issue
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_lo(tmem + Cfg::kColDP, dV_k + kstep(kk), dDO_k + kstep(kk), idSS, kk > 0);
          tc_commit(bar(C_DPFULL));
          BD_TRACE_EVENT(3, int(sc));  // MMA: waits P
          if (!(ok = mbar_wait(bar(C_PREADY), sc & 1, abort_flag))) break;
          // a unit's first dV / dK overwrite the accumulators the previous unit's
          // epilogue reads out of TMEM
          if (s == 0 && !(ok = mbar_wait(bar(C_DVFREE), (u & 1) ^ 1, abort_flag))) break;
          BD_TRACE_EVENT(4, int(sc));  // MMA: dV issue
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_lo(tmem + Cfg::kColDV, tmem + (kk >> 2) * 64 + (kk & 3) * 8, dDO_mn + mnstep(kk), idKM,
                   (s > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(C_DOEMPTY));
          // the next step's scores go ahead of this step's dK / dQ so that the
          // P^T warps can start on them while the tensor core finishes this step
          // (P^T of this step, in the same TMEM columns, was read by dV above)
          if (s + 1 < nsteps) {
            if (!(ok = mbar_wait(bar(C_QFULL0 + ((sc + 1) & 1)), ((sc + 1) >> 1) & 1, abort_flag))) break;
            tc_fence_after();
            issue_s(sc + 1);
          }
          BD_TRACE_EVENT(5, int(sc));  // MMA: waits dS
          if (!(ok = mbar_wait(bar(C_DSREADY), sc & 1, abort_flag))) break;
          BD_TRACE_EVENT(6, int(sc));  // MMA: dQ/dK issue
          if (s == 0 && !(ok = mbar_wait(bar(C_DKFREE), (u & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          // dQ first: its drain gates the next step's dP^T (same TMEM columns)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_lo(tmem + Cfg::kColDP, dDS_mn + mnstep(kk), dK_mn + mnstep(kk), idMM, kk > 0);
          tc_commit(bar(C_DQFULL));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_lo(tmem + Cfg::kColDK, dDS_k + kstep(kk), dQ_mn(qs) + mnstep(kk), idKM, (s > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(C_QEMPTY0 + qs));  // Q and dS^T of this step are free after dK
          BD_TRACE_EVENT(7, int(sc));  // MMA: dK issued
          if (s == nsteps - 1) {
            tc_commit(bar(C_ACCDONE));
            tc_commit(bar(C_KVEMPTY));
          }
        }
        ++u;
      }
      if (!ok) {
        tc_commit(bar(C_DRAIN));
        mbar_wait_drain(bar(C_DRAIN), 0);
      }
    }
   }
  } else if (warp < 12) {
    regs_set<Cfg::kRegsCompute, Cfg::kRegsLaunch>();
    // ------------------------------------------------------------ P^T / dS^T
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int jl = quarter * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t sc = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      const int w = unit_take(bar(C_UFULL), bar(C_UEMPTY), unit_ring, uk, abort_flag, false);
      if (w == -2) ok = false;
      if (w < 0) break;
      const int32_t* W = work + w * kBwdWords;
      if (W[W_NQ] == 0) continue;
      const int j = W[W_KEY0] + jl;  // global key row
      const StepRange<128> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
      for (int it = R.it_lo; it < R.it_hi && ok; ++it) {
        int t0, t1, r0;
        if (!R.tiles(it, t0, t1, r0)) continue;
        const uint32_t bseq = uint32_t(items[it * kItemWords + I_B]);
        for (int t = t0; t <= t1 && ok; ++t)
          for (int hh = 0; hh < a.G && ok; ++hh, ++sc) {
            const int qs = sc & 1;
            const uint32_t hq = uint32_t(W[W_G] * a.G + hh);  // query head
            const int i0 = r0 + t * 128;  // global row of query column 0
            const float* st_lse = reinterpret_cast<const float*>(smem + Cfg::kOffStat + qs * Cfg::kStatBytes);
            const float* st_d = st_lse + 128;
            // the query rows' document starts come from global memory (the plan),
            // read before the waits so that their latency hides behind them: the last
            // row's for the whole-tile test, and lane l's row of each 32-column chunk
            // for masking (shared with the other lanes by shuffles)
            const int32_t* g_ds = a.rowds + int64_t(it) * a.Lpad + t * 128;
            const int ds_last = __ldg(g_ds + 127);
            const int ds_mine0 = __ldg(g_ds + half * 64 + lane), ds_mine1 = __ldg(g_ds + half * 64 + 32 + lane);
            if (!(ok = mbar_wait(bar(C_QFULL0 + qs), (sc >> 1) & 1, abort_flag))) break;
            if (threadIdx.x == 128) BD_TRACE_EVENT(10, int(sc));  // compute: waits S
            if (!(ok = mbar_wait(bar(C_SFULL), sc & 1, abort_flag))) break;
            if (threadIdx.x == 128) BD_TRACE_EVENT(11, int(sc));  // compute: S ready
            tc_fence_after();
            // Rows' document starts are non-decreasing and invalid rows carry
            // INT_MAX, so key j sees every query of the tile iff it lies at or
            // before the tile's first row and at or after the last row's doc start.
            const bool full = (j <= i0) && (j >= ds_last);
            // P^T is kept as the bf16 pairs written to TMEM (the dV MMA reads the same
            // rounded values); dS below unpacks them
            uint32_t pk[2][16];
            uint32_t keep[2] = {0u, 0u};  // dropout: bit e of chunk ch keeps query i0 + ib + e
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + half * 64 + ch * 32, r);
              tmem_ld_wait();
              reg_fence(r);
              const int ib = half * 64 + ch * 32;
              float p[32];
#pragma unroll
              for (int e4 = 0; e4 < 8; ++e4) {
                const float4 l4 = ld_shared_f4(st_lse + ib + 4 * e4);
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  p[4 * e4 + k] = ex2(fmaf(__uint_as_float(r[4 * e4 + k]), a.scale_log2, -lv[k]));
              }
              // (lanes are keys, so the whole-tile test differs across the warp: every
              // lane takes part in the shuffles whenever one of them masks)
              if (__any_sync(0xffffffffu, !full)) {
                // key j sees the chunk's queries e in [elo, ehi): e >= j - (i0 + ib) for
                // causality, and e < ehi where ehi counts the chunk's rows whose document
                // starts at or before j (a prefix: the starts are non-decreasing and
                // invalid rows, INT_MAX, come last), found by a binary search over the
                // starts the lanes hold (lane l: row ib + l)
                const int ds_mine = ch ? ds_mine1 : ds_mine0;
                int ehi = 0;
#pragma unroll
                for (int step = 16; step >= 1; step >>= 1)
                  if (__shfl_sync(0xffffffffu, ds_mine, ehi + step - 1) <= j) ehi += step;
                if (__shfl_sync(0xffffffffu, ds_mine, ehi) <= j) ++ehi;
                const int elo = j - (i0 + ib);
                // bit e of `seen`: key j sees query e of the chunk (one bit test per element)
                uint32_t seen = 0u;
                if (elo < ehi && elo <= 31 && ehi >= 1)
                  seen = (elo <= 0 ? 0xffffffffu : (0xffffffffu << elo)) & (ehi >= 32 ? 0xffffffffu : ((1u << ehi) - 1u));
#pragma unroll
                for (int e = 0; e < 32; ++e) p[e] = (seen & (1u << e)) ? p[e] : 0.f;
              }
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[ch][e] = pack_bf16(p[2 * e], p[2 * e + 1]);
              if constexpr (DROP) {
                // keep bits of queries ibase .. ibase + 31 for this key: one Philox call
                // per 2-query block (word 2 (i mod 2) + (j mod 2) of counter (j/2, i/2, h, b))
                const int ibase = i0 + ib;
                uint32_t kb = 0;
                if ((ibase & 1) == 0 && (W[W_KEY0] & 1) == 0) {
                  // keys 2m, 2m + 1 are lanes 2m, 2m + 1: each lane makes every other
                  // call of the pair and hands its partner the two words it needs
                  const uint32_t odd = lane & 1;
#pragma unroll
                  for (int m = 0; m < 8; ++m) {
                    const uint4 rr = philox4x32_10(
                        make_uint4(uint32_t(j) >> 1, uint32_t(ibase >> 1) + 2 * m + odd, hq, bseq), a.drop_k0,
                        a.drop_k1);
                    const uint32_t ev = uint32_t(rr.x >= a.drop_thresh) | (uint32_t(rr.z >= a.drop_thresh) << 1);
                    const uint32_t od = uint32_t(rr.y >= a.drop_thresh) | (uint32_t(rr.w >= a.drop_thresh) << 1);
                    const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? ev : od, 1);
                    const uint32_t lo = odd ? got : ev, hi = odd ? od : got;  // query blocks 2m, 2m + 1
                    kb |= (lo | (hi << 2)) << (4 * m);
                  }
                } else if ((ibase & 1) == 0) {
#pragma unroll
                  for (int e2 = 0; e2 < 16; ++e2) {
                    const uint4 rr = philox4x32_10(
                        make_uint4(uint32_t(j) >> 1, uint32_t(ibase >> 1) + e2, hq, bseq), a.drop_k0, a.drop_k1);
                    const uint32_t w0 = (j & 1) ? rr.y : rr.x, w1 = (j & 1) ? rr.w : rr.z;
                    kb |= (uint32_t(w0 >= a.drop_thresh) << (2 * e2)) | (uint32_t(w1 >= a.drop_thresh) << (2 * e2 + 1));
                  }
                } else {
#pragma unroll 4
                  for (int e = 0; e < 32; ++e) {
                    const int i = ibase + e;
                    const uint4 rr = philox4x32_10(make_uint4(uint32_t(j) >> 1, uint32_t(i) >> 1, hq, bseq),
                                                   a.drop_k0, a.drop_k1);
                    const uint32_t w = (i & 1) ? ((j & 1) ? rr.w : rr.z) : ((j & 1) ? rr.y : rr.x);
                    kb |= uint32_t(w >= a.drop_thresh) << e;
                  }
                }
                keep[ch] = kb;
                // the dV product reads the dropped, rescaled probabilities
                uint32_t pd[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  pd[e] = pack_bf16(((kb >> (2 * e)) & 1) ? p[2 * e] * a.drop_scale : 0.f,
                                    ((kb >> (2 * e + 1)) & 1) ? p[2 * e + 1] * a.drop_scale : 0.f);
                tmem_st16(tmem + lane_base + half * 64 + ch * 16, pd);
              } else {
                tmem_st16(tmem + lane_base + half * 64 + ch * 16, pk[ch]);
              }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(C_PREADY));
            if (threadIdx.x == 128) BD_TRACE_EVENT(12, int(sc));  // compute: P stored
            if (!(ok = mbar_wait(bar(C_DPFULL), sc & 1, abort_flag))) break;
            if (threadIdx.x == 128) BD_TRACE_EVENT(13, int(sc));  // compute: dP ready
            tc_fence_after();
            // dS^T of the previous step must have been consumed by its dQ and dK MMAs
            // (dK is the later one; its commit also releases that step's Q stage)
            if (sc > 0 && !(ok = mbar_wait(bar(C_QEMPTY0 + ((sc - 1) & 1)), ((sc - 1) >> 1) & 1, abort_flag)))
              break;
            const uint32_t row_addr = sDS + half * 16384 + jl * 128;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + Cfg::kColDP + half * 64 + ch * 32, r);
              tmem_ld_wait();
              reg_fence(r);
              const int ib = half * 64 + ch * 32;
              uint32_t dsk[16];
#pragma unroll
              for (int e4 = 0; e4 < 8; ++e4) {
                const float4 d4 = ld_shared_f4(st_d + ib + 4 * e4);
                const int e = 4 * e4;
                const uint32_t p01 = pk[ch][2 * e4], p23 = pk[ch][2 * e4 + 1];
                float dp[4] = {__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                               __uint_as_float(r[e + 3])};
                if constexpr (DROP) {
                  // dS = P (keep dP / (1 - p) - D) with the undropped P
#pragma unroll
                  for (int k = 0; k < 4; ++k) dp[k] = ((keep[ch] >> (e + k)) & 1) ? dp[k] * a.drop_scale : 0.f;
                }
                const float s0 = __uint_as_float(p01 << 16) * (dp[0] - d4.x);
                const float s1 = __uint_as_float(p01 & 0xffff0000u) * (dp[1] - d4.y);
                const float s2 = __uint_as_float(p23 << 16) * (dp[2] - d4.z);
                const float s3 = __uint_as_float(p23 & 0xffff0000u) * (dp[3] - d4.w);
                dsk[2 * e4] = pack_bf16(s0, s1);
                dsk[2 * e4 + 1] = pack_bf16(s2, s3);
              }
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int chunk = ch * 4 + c4;  // 16-byte chunk of the 128-byte row
                st_shared_v4(row_addr + ((chunk ^ (jl & 7)) << 4), dsk[4 * c4], dsk[4 * c4 + 1], dsk[4 * c4 + 2],
                             dsk[4 * c4 + 3]);
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(C_DSREADY));
            if (threadIdx.x == 128) BD_TRACE_EVENT(14, int(sc));  // compute: dS stored
          }
      }
    }
  } else {
    regs_set<Cfg::kRegsDq, Cfg::kRegsLaunch>();
    // ------------------------------------------------------------ dQ out, dK/dV epilogue
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // query row (dQ) or key row (dK/dV) == TMEM lane
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t u = 0, sc = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      const int w = unit_take(bar(C_UFULL), bar(C_UEMPTY), unit_ring, uk, abort_flag, false);
      if (w == -2) ok = false;
      if (w < 0) break;
      const int32_t* W = work + w * kBwdWords;
      const int g = W[W_G], ob = W[W_OBUF] / a.ck_out, oc = W[W_OBUF] % a.ck_out;
      const int brow = W[W_OROW] + rl;  // output row of this lane's key
      float* dkrow = a.dk + ob * a.k_sb + oc * a.k_sc + int64_t(brow) * a.k_sr + int64_t(g) * a.k_sh;
      float* dvrow = a.dv + ob * a.v_sb + oc * a.v_sc + int64_t(brow) * a.v_sr + int64_t(g) * a.v_sh;
      const bool krow_ok = brow < a.dk_rows;
      if (W[W_NQ] == 0) {
        if (krow_ok && !a.accumulate) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int k = 0; k < D / 4; ++k) {
            reinterpret_cast<float4*>(dkrow)[k] = z;
            reinterpret_cast<float4*>(dvrow)[k] = z;
          }
        }
        continue;
      }
      const StepRange<128> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
      for (int it = R.it_lo; it < R.it_hi && ok; ++it) {
        int t0, t1, r0;
        if (!R.tiles(it, t0, t1, r0)) continue;
        const int32_t* I = items + it * kItemWords;
        const int b = I[I_B], c = I[I_C], svalid = I[I_SVALID];
        for (int t = t0; t <= t1 && ok; ++t)
          for (int hh = 0; hh < a.G && ok; ++hh, ++sc) {
            const int h = g * a.G + hh;
            const int lrow = t * 128 + rl;
            // the warpgroup meets at named barriers below: leave together or not at all
            if (rl == 0) BD_TRACE_EVENT(20, int(sc));  // dQ: waits dQ
            ok = bar_red_and(1, 128, mbar_wait(bar(C_DQFULL), sc & 1, abort_flag));
            if (rl == 0) BD_TRACE_EVENT(21, int(sc));  // dQ: dQ ready
            if (!ok) break;
            tc_fence_after();
            // dQ tile (128 query rows x D fp32) goes to global memory as TMA
            // reduce-adds (rows past L are clipped by the map); the whole dQ row
            // leaves TMEM first, so the next dP^T can start at once
            uint32_t r[D / 32][32];
#pragma unroll
            for (int q = 0; q < D / 32; ++q) tmem_ld32(tmem + lane_base + Cfg::kColDP + q * 32, r[q]);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < D / 32; ++q) reg_fence(r[q]);
            tc_fence_before();
            mbar_arrive(bar(C_DQEMPTY));
            if (rl == 0) BD_TRACE_EVENT(22, int(sc));  // dQ: TMEM released
            // D/32 rounds of 128 rows x 32 columns (16 KB) through two staging buffers
            // (128-byte swizzle: 16-byte chunk c of row r sits at c ^ (r & 7)), so that
            // filling one buffer overlaps the TMA reading the other
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
              const uint32_t buf = sStage + (q & 1) * Cfg::kStageBytes;
              if (rl == 0) bulk_wait_read<1>();  // the box sent from this buffer two rounds ago has left it
              named_bar_sync(1, 128);
              const uint32_t* v = r[q];
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4)
                st_shared_v4(buf + rl * 128 + ((c4 ^ (rl & 7)) << 4),
                             __float_as_uint(__uint_as_float(v[4 * c4]) * a.scale),
                             __float_as_uint(__uint_as_float(v[4 * c4 + 1]) * a.scale),
                             __float_as_uint(__uint_as_float(v[4 * c4 + 2]) * a.scale),
                             __float_as_uint(__uint_as_float(v[4 * c4 + 3]) * a.scale));
              fence_proxy_async_smem();
              named_bar_sync(1, 128);
              if (rl == 0) {
                tma_reduce_add_5d(&tm_dq, buf, q * 32, h, t * 128, c, b);
                bulk_commit();
              }
            }
            (void)lrow;
            (void)svalid;
          }
      }
      if (!ok) break;
      // the warpgroup meets at named barriers below when TMA takes the rows out
      ok = bar_red_and(1, 128, mbar_wait(bar(C_ACCDONE), u & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      // dV, then dK (x scale), each leaving TMEM whole first (so that the next
      // unit's first dV / dK MMA can start), go out as 128-row x 32-column boxes
      // through the two staging buffers, stored (or added) by TMA: one thread's
      // row per lane written 32 bytes at a time by the load/store unit kept it busy
      // for ~9k cycles a unit, stalling the next unit's loads
#pragma unroll 1
      for (int x = 0; x < 2; ++x) {
        uint32_t v[D / 32][32];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tmem_ld32(tmem + lane_base + (x ? Cfg::kColDK : Cfg::kColDV) + q * 32, v[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < D / 32; ++q) reg_fence(v[q]);
        tc_fence_before();
        mbar_arrive(bar(x ? C_DKFREE : C_DVFREE));
        const float mul = x ? a.scale : 1.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          const uint32_t buf = sStage + (q & 1) * Cfg::kStageBytes;
          if (rl == 0) bulk_wait_read<1>();  // the box sent from this buffer two rounds ago has left it
          named_bar_sync(1, 128);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            st_shared_v4(buf + rl * 128 + ((c4 ^ (rl & 7)) << 4),
                         __float_as_uint(__uint_as_float(v[q][4 * c4]) * mul),
                         __float_as_uint(__uint_as_float(v[q][4 * c4 + 1]) * mul),
                         __float_as_uint(__uint_as_float(v[q][4 * c4 + 2]) * mul),
                         __float_as_uint(__uint_as_float(v[q][4 * c4 + 3]) * mul));
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (rl == 0) {
            const CUtensorMap* m = x ? &tm_dk : &tm_dv;
            if (a.accumulate) tma_reduce_add_5d(m, buf, q * 32, g, W[W_OROW], oc, ob);
            else tma_store_5d(m, buf, q * 32, g, W[W_OROW], oc, ob);
            bulk_commit();
          }
        }
      }
      ++u;
    }
    if (rl == 0) bulk_wait<0>();  // every dQ reduce-add has completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    if (*abort_flag) {
      atomicExch(const_cast<int32_t*>(plan) + H_STATUS, DEV_TIMEOUT);
      atomicExch(const_cast<int32_t*>(plan) + H_STATUS_DETAIL, 2);
    }
    unit_counters_release(claim, claim + 1);
  }
}

template <int D, bool DROP>
static int32_t launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                          const CUtensorMap& mdo, const CUtensorMap& mdq, const CUtensorMap& mdk,
                          const CUtensorMap& mdv, const BwdArgs& a, int grid, cudaStream_t stream) {
  using Cfg = BwdCfg<D>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bd_bwd_kernel<D, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, bd_bwd_kernel<D, DROP>);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(bwd)");
    // the setmaxnreg directions were chosen for this launch count: refuse any other
    if (fa.numRegs != Cfg::kRegsLaunch)
      return fail(BD_ERR_UNSUPPORTED, "bwd kernel built with %d registers/thread, its register split assumes %d",
                  fa.numRegs, Cfg::kRegsLaunch);
    attr_done[dev] = true;
  }
  bd_bwd_kernel<D, DROP><<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(mq, mk, mv, mdo, mdq, mdk, mdv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bd_bwd_kernel launch");
  return BD_OK;
}

}  // namespace bd

using namespace bd;

#ifdef BD_TRACE
// Trace build only: the backward kernel's [site][tile] clock table of CTA 0.
extern "C" BD_API int32_t bd_trace_read_bwd(unsigned long long* host, int32_t cap) {
  const int32_t n = dev::kTraceSites * dev::kTraceTiles;
  const int32_t k = n < cap ? n : cap;
  cudaDeviceSynchronize();
  if (k > 0) cudaMemcpyFromSymbol(host, dev::g_bd_trace, size_t(k) * 8);
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, dev::g_bd_trace) == cudaSuccess) cudaMemset(p, 0, size_t(n) * 8);
  cudaDeviceSynchronize();
  return k;
}
#endif

extern "C" int32_t bd_attn_bwd_workspace(const void* plan_host, size_t* bytes) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!bytes) return fail(BD_ERR_ARG, "bytes is NULL");
  *bytes = bwd_workspace_layout(pv.hdr(H_NITEMS), pv.hdr(H_H), pv.hdr(H_QTILES) * 128).total;
  return ok();
}

namespace {

struct BwdCommon {
  PlanView pv;
  int B, C, L, H, Hkv, D, Ck, nitems, Lpad;
  BwdWorkspace ws;
};

int32_t bwd_common(const void* plan_host, const void* plan_dev, void* workspace, size_t workspace_bytes,
                   BwdCommon* c) {
  int32_t st = view_plan(plan_host, &c->pv);
  if (st) return st;
  if (!plan_dev || reinterpret_cast<uintptr_t>(plan_dev) % 16)
    return fail(BD_ERR_ARG, "plan_dev NULL or not 16-byte aligned");
  const PlanView& pv = c->pv;
  c->B = pv.hdr(H_B); c->C = pv.hdr(H_C); c->L = pv.hdr(H_L); c->H = pv.hdr(H_H); c->Hkv = pv.hdr(H_HKV);
  c->D = pv.hdr(H_D); c->Ck = pv.hdr(H_CK); c->nitems = pv.hdr(H_NITEMS); c->Lpad = pv.hdr(H_QTILES) * 128;
  if (c->D != 64 && c->D != 128 && c->D != 256)
    return fail(BD_ERR_UNSUPPORTED, "the backward supports head dim 64, 128 and 256; this plan has %d", c->D);
  c->ws = bwd_workspace_layout(c->nitems, c->H, c->Lpad);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(BD_ERR_ALIGN, "workspace NULL or not 256-byte aligned");
  if (workspace_bytes < c->ws.total) return fail(BD_ERR_CAPACITY, "workspace needs %zu bytes", c->ws.total);
  return BD_OK;
}

}  // namespace

extern "C" int32_t bd_attn_bwd_pre_ex(const void* plan_host, const void* plan_dev, const bd_tensor* out,
                                      const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq, void* workspace,
                                      size_t workspace_bytes, int32_t clear_dq, void* stream) {
  BwdCommon c;
  int32_t st = bwd_common(plan_host, plan_dev, workspace, workspace_bytes, &c);
  if (st) return st;
  if ((st = check_tensor(out, "out", 2, c.B, c.C, c.H, true))) return st;
  if ((st = check_tensor(dout, "dout", 2, c.B, c.C, c.H, true))) return st;
  if ((st = check_tensor(dq, "dq", 4, c.B, c.C, c.H, false))) return st;
  if (out->rows != c.L || dout->rows != c.L || dq->rows != c.L)
    return fail(BD_ERR_ARG, "out/dout/dq rows must equal L = %d", c.L);
  if (!lse || !lse->ptr || reinterpret_cast<uintptr_t>(lse->ptr) % 4) return fail(BD_ERR_ARG, "lse NULL/misaligned");
  char* wsb = static_cast<char*>(workspace);
  BwdPreArgs p;
  p.plan = static_cast<const int32_t*>(plan_dev);
  p.lse = lse->ptr; p.l_sb = lse->stride_b; p.l_sc = lse->stride_c; p.l_sh = lse->stride_head;
  p.lse2 = reinterpret_cast<float*>(wsb + c.ws.lse2);
  p.dstat = reinterpret_cast<float*>(wsb + c.ws.dstat);
  p.counters = reinterpret_cast<int32_t*>(wsb + c.ws.counters);
  p.dq = static_cast<float*>(dq->ptr);
  p.q_sb = dq->stride_b; p.q_sc = dq->stride_c; p.q_sr = dq->stride_row; p.q_sh = dq->stride_head;
  p.nitems = c.nitems; p.C = c.C; p.L = c.L; p.Lpad = c.Lpad; p.H = c.H; p.clear_dq = clear_dq ? 1 : 0;
  p.items_off = c.pv.hdr(H_OFF_ITEMS);
  {
    // a group (one shared-memory box of O, one of dO: 8 KB each) holds whole
    // head-rows: up to 4096 / d heads of a power-of-two number of rows (<= 128,
    // so that groups tile Lpad)
    p.heads = std::min(c.H, 4096 / c.D);
    int rows = 1;
    while (rows < 128 && 2 * rows * p.heads * c.D * 2 <= 8192) rows *= 2;
    p.rows = rows;
    p.head_blocks = (c.H + p.heads - 1) / p.heads;
    const int64_t ngroups = int64_t(c.nitems) * (c.Lpad / rows) * p.head_blocks;
    if (ngroups > 0x7fffffff) return fail(BD_ERR_UNSUPPORTED, "too many rows for the statistics kernel");
    p.ngroups = int32_t(ngroups);
  }
  CUtensorMap mo, mdo;
  if ((st = make_tmap_rows_bf16(&mo, out, c.B, c.C, c.H, c.D, "out", p.heads, p.rows))) return st;
  if ((st = make_tmap_rows_bf16(&mdo, dout, c.B, c.C, c.H, c.D, "dout", p.heads, p.rows))) return st;
  if ((st = launch_bwd_pre(mo, mdo, p, c.D, static_cast<cudaStream_t>(stream)))) return st;
  return ok();
}

extern "C" int32_t bd_attn_bwd_pre(const void* plan_host, const void* plan_dev, const bd_tensor* out,
                                   const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return bd_attn_bwd_pre_ex(plan_host, plan_dev, out, dout, lse, dq, workspace, workspace_bytes, 1, stream);
}

namespace {

// The main backward kernel over the plan's main work list (dK / dV into the
// K/V-buffer-shaped dk / dv) or, with owner set, over its owner list (dK / dV
// of every chunk summed into owner-row tensors [B, 1, S, Hkv, d]).
int32_t bwd_main_impl(const void* plan_host, const void* plan_dev, const bd_tensor* q, const bd_tensor* k,
                      const bd_tensor* v, const bd_tensor* dout, bd_tensor* dq, bd_tensor* dk, bd_tensor* dv,
                      int32_t accumulate_dkv, void* workspace, size_t workspace_bytes, void* stream, bool owner,
                      bool launch = true) {
  BwdCommon c;
  int32_t st = bwd_common(plan_host, plan_dev, workspace, workspace_bytes, &c);
  if (st) return st;
  const PlanView& pv = c.pv;
  if (owner && pv.hdr(H_NBWDO) == 0)
    return fail(BD_ERR_UNSUPPORTED,
                "the plan has no owner-keyed backward work: it needs BD_KV_WINDOW, every chunk 0..cp-1 in "
                "order and L a multiple of 128");
  const int ck_out = owner ? 1 : c.Ck;
  if ((st = check_tensor(q, "q", 2, c.B, c.C, c.H, true))) return st;
  if ((st = check_tensor(dout, "dout", 2, c.B, c.C, c.H, true))) return st;
  if ((st = check_tensor(k, "k", 2, c.B, c.Ck, c.Hkv, true))) return st;
  if ((st = check_tensor(v, "v", 2, c.B, c.Ck, c.Hkv, true))) return st;
  if ((st = check_tensor(dq, "dq", 4, c.B, c.C, c.H, true))) return st;
  if ((st = check_tensor(dk, "dk", 4, c.B, ck_out, c.Hkv, false))) return st;
  if ((st = check_tensor(dv, "dv", 4, c.B, ck_out, c.Hkv, false))) return st;
  if (q->rows != c.L || dout->rows != c.L || dq->rows != c.L)
    return fail(BD_ERR_ARG, "q/dout/dq rows must equal L = %d", c.L);
  if (k->rows < pv.hdr(H_KV_ROWS) || v->rows < pv.hdr(H_KV_ROWS))
    return fail(BD_ERR_ARG, "k/v rows < %d needed by the plan", pv.hdr(H_KV_ROWS));
  if (dk->rows != dv->rows) return fail(BD_ERR_ARG, "dk and dv must have the same rows");
  if (owner) {
    if (dk->rows < pv.hdr(H_S)) return fail(BD_ERR_ARG, "owner dk/dv rows must be >= S = %d", pv.hdr(H_S));
  } else if (dk->rows < pv.hdr(H_KV_ROWS)) {
    return fail(BD_ERR_ARG, "dk/dv rows < %d", pv.hdr(H_KV_ROWS));
  }
  CUtensorMap mq, mk, mv, mdo, mdq;
  // dQ reduce boxes: 128 rows x 32 columns (128-byte swizzle), or at head dim 256
  // (transposed dQ) 16 rows x 32 columns; Q / dO boxes are one backward query
  // step high
  if ((st = c.D == 256 ? make_tmap_f32_reduce(&mdq, dq, c.B, c.C, c.H, c.D, "dq", 128, 16)
                       : make_tmap_f32_reduce(&mdq, dq, c.B, c.C, c.H, c.D, "dq", 32, 128)))
    return st;
  if ((st = make_tmap_bf16(&mq, q, c.B, c.C, c.H, c.D, "q", bwd_query_step(c.D)))) return st;
  if ((st = make_tmap_bf16(&mdo, dout, c.B, c.C, c.H, c.D, "dout", bwd_query_step(c.D)))) return st;
  if ((st = make_tmap_bf16(&mk, k, c.B, c.Ck, c.Hkv, c.D, "k"))) return st;
  if ((st = make_tmap_bf16(&mv, v, c.B, c.Ck, c.Hkv, c.D, "v"))) return st;
  char* wsb = static_cast<char*>(workspace);
  BwdArgs a;
  a.plan = static_cast<const int32_t*>(plan_dev);
  a.lse2 = reinterpret_cast<const float*>(wsb + c.ws.lse2);
  a.dstat = reinterpret_cast<const float*>(wsb + c.ws.dstat);
  a.rowds = static_cast<const int32_t*>(plan_dev) + pv.hdr(H_OFF_ROWDS);
  a.counters = reinterpret_cast<int32_t*>(wsb + c.ws.counters);
  a.dq = static_cast<float*>(dq->ptr);
  a.q_sb = dq->stride_b; a.q_sc = dq->stride_c; a.q_sr = dq->stride_row; a.q_sh = dq->stride_head;
  a.dk = static_cast<float*>(dk->ptr);
  a.k_sb = dk->stride_b; a.k_sc = dk->stride_c; a.k_sr = dk->stride_row; a.k_sh = dk->stride_head;
  a.dv = static_cast<float*>(dv->ptr);
  a.v_sb = dv->stride_b; a.v_sc = dv->stride_c; a.v_sr = dv->stride_row; a.v_sh = dv->stride_head;
  a.L = c.L; a.Lpad = c.Lpad; a.H = c.H; a.G = pv.hdr(H_G); a.Ck = c.Ck;
  a.n_work = owner ? pv.hdr(H_NBWDO) : pv.hdr(H_NBWD);
  a.work_off = owner ? pv.hdr(H_OFF_BWDO) : pv.hdr(H_OFF_BWD);
  a.ck_out = ck_out;
  a.accumulate = accumulate_dkv ? 1 : 0; a.dk_rows = dk->rows;
  // dK / dV leave by TMA in 128-row x 32-column fp32 boxes (the checks above give
  // the 16-byte aligned base and strides a tensor map needs)
  CUtensorMap mdk, mdv;
  std::memset(&mdk, 0, sizeof(mdk));
  std::memset(&mdv, 0, sizeof(mdv));
  if (c.D != 256) {
    if ((st = make_tmap_f32_reduce(&mdk, dk, c.B, ck_out, c.Hkv, c.D, "dk", 32, 128))) return st;
    if ((st = make_tmap_f32_reduce(&mdv, dv, c.B, ck_out, c.Hkv, c.D, "dv", 32, 128))) return st;
  }
  float scale;
  const int32_t sb = pv.hdr(H_SCALE_BITS);
  memcpy(&scale, &sb, 4);
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  if (!launch || a.n_work == 0) return ok();  // validation only, or nothing to do
  int nsm = 0;
  if ((st = sm_count(&nsm))) return st;
  const int grid = a.n_work < nsm ? a.n_work : nsm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  a.drop_thresh = uint32_t(pv.hdr(H_DROP_THRESH));
  a.drop_k0 = uint32_t(pv.hdr(H_DROP_SEED_LO));
  a.drop_k1 = uint32_t(pv.hdr(H_DROP_SEED_HI));
  const int32_t dbits = pv.hdr(H_DROP_SCALE_BITS);
  memcpy(&a.drop_scale, &dbits, 4);
  if (c.D == 256)
    st = launch_bwd256(mq, mk, mv, mdo, mdq, a, a.drop_thresh != 0, grid, s);
  else if (a.drop_thresh != 0)
    st = c.D == 128 ? launch_bwd<128, true>(mq, mk, mv, mdo, mdq, mdk, mdv, a, grid, s)
                    : launch_bwd<64, true>(mq, mk, mv, mdo, mdq, mdk, mdv, a, grid, s);
  else
    st = c.D == 128 ? launch_bwd<128, false>(mq, mk, mv, mdo, mdq, mdk, mdv, a, grid, s)
                    : launch_bwd<64, false>(mq, mk, mv, mdo, mdq, mdk, mdv, a, grid, s);
  if (st) return st;
  return ok();
}

}  // namespace

extern "C" int32_t bd_attn_bwd_main(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                                    const bd_tensor* k, const bd_tensor* v, const bd_tensor* dout, bd_tensor* dq,
                                    bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return bwd_main_impl(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace, workspace_bytes,
                       stream, false);
}

extern "C" int32_t bd_attn_bwd_main_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                                       const bd_tensor* k, const bd_tensor* v, const bd_tensor* dout, bd_tensor* dq,
                                       bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, int32_t flags,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  if (flags & ~int32_t(BD_BWD_OWNER_ROWS | BD_BWD_DQ_ZEROED)) return fail(BD_ERR_ARG, "unknown flags 0x%x", flags);
  return bwd_main_impl(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace, workspace_bytes,
                       stream, (flags & BD_BWD_OWNER_ROWS) != 0);
}

extern "C" int32_t bd_attn_bwd(const void* plan_host, const void* plan_dev, const bd_tensor* q, const bd_tensor* k,
                               const bd_tensor* v, const bd_tensor* out, const bd_tensor* dout,
                               const bd_rowstat* lse, bd_tensor* dq, bd_tensor* dk, bd_tensor* dv,
                               int32_t accumulate_dkv, void* workspace, size_t workspace_bytes, void* stream) {
  // the main step's arguments are checked before the statistics kernel runs
  int32_t st = bwd_main_impl(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace,
                             workspace_bytes, stream, false, false);
  if (st) return st;
  st = bd_attn_bwd_pre(plan_host, plan_dev, out, dout, lse, dq, workspace, workspace_bytes, stream);
  if (st) return st;
  return bd_attn_bwd_main(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace,
                          workspace_bytes, stream);
}

extern "C" int32_t bd_attn_bwd_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                                  const bd_tensor* k, const bd_tensor* v, const bd_tensor* out, const bd_tensor* dout,
                                  const bd_rowstat* lse, bd_tensor* dq, bd_tensor* dk, bd_tensor* dv,
                                  int32_t accumulate_dkv, int32_t flags, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (flags & ~int32_t(BD_BWD_OWNER_ROWS | BD_BWD_DQ_ZEROED)) return fail(BD_ERR_ARG, "unknown flags 0x%x", flags);
  const bool owner = (flags & BD_BWD_OWNER_ROWS) != 0;
  // the main step's arguments (and, for owner rows, the plan's owner list) are
  // checked before the statistics kernel runs
  int32_t st = bwd_main_impl(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace,
                             workspace_bytes, stream, owner, false);
  if (st) return st;
  st = bd_attn_bwd_pre_ex(plan_host, plan_dev, out, dout, lse, dq, workspace, workspace_bytes,
                          (flags & BD_BWD_DQ_ZEROED) ? 0 : 1, stream);
  if (st) return st;
  return bwd_main_impl(plan_host, plan_dev, q, k, v, dout, dq, dk, dv, accumulate_dkv, workspace, workspace_bytes,
                       stream, owner);
}
