// Backward of block-causal varlen chunked attention at head dim 256 on sm_103a.
//
// Same gradients as the head dim 64 / 128 kernel (the analytic gradient of the
// forward of the NeMo Automodel page "block-diagonal varlen CP for packed
// sequences", Design overview): P = exp(scale q k - LSE) on the block-causal
// mask, dV = P^T dO, dP = dO V^T, dS = P (dP - D), dQ = scale dS K,
// dK = scale dS^T Q, dK/dV summed over the query heads of a GQA group.
//
// At head dim 256 the 128-key tile's dK and dV accumulators (128 x 256 fp32 each)
// would take all 512 TMEM columns, and a 128-row Q tile plus dO tile (64 KB
// each) would not fit in shared memory beside the resident K and V tiles
// (64 KB each). So a work unit (one 128-row K/V tile of one K/V head) is walked
// twice:
//   pass 0  S^T = K Q^T, P^T, dV += P^T dO            (dV in TMEM columns 256..511)
//           in 128-row query steps: V is not needed yet, so its place holds the
//           128-row Q tile and V is loaded for pass 1; S^T alternates between
//           TMEM columns 0..127 and 128..255, so the next step's S^T runs while
//           this step's P^T is formed
//   pass 1  S^T, dP^T = V dO^T, dS^T, dK += dS^T Q,   (dK in the same columns)
//           dQ^T = K^T dS^T (two 128-row halves of d), in 64-row query steps
// S^T is recomputed in pass 1; every other product is formed once. Pass 1 walks
// the steps in reverse order, so that it starts on the Q / dO tiles pass 0 read
// last, which are the ones still in L2.
// Roles (16 warps, one persistent CTA per SM claiming units dynamically):
//   warp 0       TMA producer: K/V once per unit; per step the Q and dO tiles
//                (64 rows x 256) and, into a two-stage ring of their own, the
//                step's row statistics (LSE, D, document start).
//   warp 1       TMEM allocation; one thread issues the MMAs.
//   warps 4-11   P^T (pass 0, into TMEM for the dV product) and dS^T (pass 1,
//                into shared memory), lane = key row, 32 queries per warp.
//   warps 12-15  pass 1: read dQ^T (lane = column of d) out of TMEM, transpose it
//                through two shared staging boxes (16 query rows x one d half)
//                and add it into dQ with TMA reduce-adds; end of each pass:
//                write dV, then dK (x scale).
// TMEM columns: S^T [0, 64), dP^T [64, 128), dQ^T [128, 256), dV / dK [256, 512).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd_kernel.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace bd {
using namespace dev;

namespace {

struct Cfg256 {
  static constexpr int D = 256, QR = 64;        // head dim, query rows per step
  static constexpr int kKVBytes = 128 * D * 2;  // one K or V tile: four 128-row x 64-column boxes
  static constexpr int kQBox = QR * 128;        // one 64-row x 64-column box of a Q / dO tile
  static constexpr int kQBytes = QR * D * 2;
  static constexpr int kOffK = 0, kOffV = kKVBytes, kOffQ = 2 * kKVBytes;
  static constexpr int kOffDO = kOffQ + kQBytes;
  static constexpr int kOffDS = kOffDO + kQBytes;      // dS^T: 128 keys x 64 queries bf16
  static constexpr int kOffStage = kOffDS + 128 * QR * 2;  // dQ staging: two 16-row x 128-column fp32 boxes
  static constexpr int kStageBytes = 16384;
  static constexpr int kOffStat = kOffStage + kStageBytes;  // two stages: lse2, D, ds of 64 rows
  static constexpr int kStatBytes = 3 * QR * 4;
  static constexpr int kOffBar = kOffStat + 2 * kStatBytes;
  static constexpr int kSmem = kOffBar + 512 + 1024;
  // pass 0 (no V resident): 128-row Q tiles in V's place, 128-row dO tiles across the
  // Q and dO places, and their row statistics (two stages) in the dS^T place
  static constexpr int kOffQ0 = kOffV, kOffDO0 = kOffQ;
  static constexpr int kStat0Bytes = 3 * 128 * 4;
  static_assert(kOffDO == kOffQ + kQBytes && 2 * kQBytes == kKVBytes, "the 128-row dO tile spans the Q and dO places");
  static_assert(2 * kStat0Bytes <= 128 * QR * 2, "pass-0 statistics exceed the dS^T place");
  static constexpr int kColS = 0, kColDP = 64, kColDQ = 128, kColAcc = 256;
  static constexpr int kThreads = 512;
  static constexpr int kRegsCtl = 96, kRegsCompute = 120, kRegsDq = 176, kRegsLaunch = 128;
  static_assert(128 * kRegsCtl + 256 * kRegsCompute + 128 * kRegsDq <= kRegsLaunch * kThreads,
                "register split exceeds the launch's registers");
  static_assert(kSmem <= 232448, "shared memory beyond the 227 KB a CTA may have");
  static_assert(kOffStage % 1024 == 0, "staging boxes need 1024-byte alignment for the 128-byte swizzle");
};

enum : int {
  E_KVFULL = 0, E_KVEMPTY, E_QFULL, E_QEMPTY, E_DOFULL, E_DOEMPTY, E_SFULL, E_DPFULL, E_PREADY0, E_PREADY1, E_DSREADY,
  E_DQFULL, E_DQEMPTY, E_DSFREE, E_ACCDONE, E_ACCFREE, E_DRAIN, E_STFULL0, E_STFULL1, E_STEMPTY0, E_STEMPTY1,
  E_VFULL, E_S0FULL0, E_S0FULL1, E_UFULL, E_UEMPTY = E_UFULL + kUnitSlots, E_COUNT = E_UEMPTY + kUnitSlots
};
constexpr uint32_t kConsumers256 = 1 + 8 + 4;  // MMA thread, 8 P/dS warps, 4 dQ warps
static_assert(8 * E_COUNT + 16 + 4 * kUnitSlots <= 512, "barriers, TMEM slot, abort flag and unit ring overflow");

template <bool DROP>
__global__ void __launch_bounds__(512, 1)
    bd_bwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using C = Cfg256;
  constexpr int QR = C::QR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ, sDO = sbase + C::kOffDO;
  const uint32_t sDS = sbase + C::kOffDS, sStage = sbase + C::kOffStage;
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * E_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * E_COUNT + 8);
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + C::kOffBar + 8 * E_COUNT + 16);
  int* claim = a.counters;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t* plan = a.plan;
  const int32_t* work = plan + a.work_off;
  const int32_t* items = plan + plan[H_OFF_ITEMS];

  if (threadIdx.x == 0) {
    for (int i = 0; i < E_COUNT; ++i) {
      const uint32_t n = (i == E_PREADY0 || i == E_PREADY1 || i == E_DSREADY || i == E_STEMPTY0 || i == E_STEMPTY1) ? 256u
                         : (i == E_DQEMPTY || i == E_ACCFREE)                                   ? 128u
                         : (i >= E_UEMPTY && i < E_UEMPTY + kUnitSlots)                         ? kConsumers256
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

  if (warp < 4) {
    regs_set<C::kRegsCtl, C::kRegsLaunch>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (elect_one()) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        uint32_t u = 0, sc = 0, st_iss = 0, q_iss = 0, do_iss = 0, v_iss = 0;
        bool ok = true;
        for (uint32_t uk = 0; ok; ++uk) {
          const int w = unit_publish(bar(E_UFULL), bar(E_UEMPTY), unit_ring, claim, a.n_work, uk, abort_flag);
          if (w == -2) ok = false;
          if (w < 0) break;
          const int32_t* W = work + w * kBwdWords;
          if (W[W_NQ] == 0) continue;
          const int g = W[W_G], kb = W[W_BUF] / a.Ck, kc = W[W_BUF] % a.Ck;
          // K for both passes (the previous unit's last products have read K and V)
          if (!(ok = mbar_wait(bar(E_KVEMPTY), (u & 1) ^ 1, abort_flag))) break;
          mbar_expect_tx(bar(E_KVFULL), C::kKVBytes);
          for (int hf = 0; hf < 4; ++hf)
            tma_load_5d(sK + hf * 16384, &tm_k, bar(E_KVFULL), hf * 64, g, W[W_LROW], kc, kb);
          ++u;
          // pass 0: 128-row steps; Q in V's place, dO across the Q and dO places (each
          // 64-column box of 128 rows loaded as two 64-row boxes), statistics of the
          // 128 rows in the dS^T place
          {
            const StepRange<128> R0{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
            for (int it = R0.it_lo; it < R0.it_hi && ok; ++it) {
              int t0, t1, r0;
              if (!R0.tiles(it, t0, t1, r0)) continue;
              const int32_t* I = items + it * kItemWords;
              const int b = I[I_B], c = I[I_C];
              for (int t = t0; t <= t1 && ok; ++t)
                for (int hh = 0; hh < a.G && ok; ++hh, ++sc) {
                  const int h = g * a.G + hh;
                  const int ss = sc & 1;
                  if (!(ok = mbar_wait(bar(E_STEMPTY0 + ss), ((sc >> 1) & 1) ^ 1, abort_flag))) break;
                  mbar_expect_tx(bar(E_STFULL0 + ss), C::kStat0Bytes);
                  const uint32_t st = sbase + C::kOffDS + ss * C::kStat0Bytes;
                  const int64_t srow = (int64_t(it) * a.H + h) * a.Lpad + t * 128;
                  bulk_load(st, a.lse2 + srow, 512, bar(E_STFULL0 + ss));
                  bulk_load(st + 512, a.dstat + srow, 512, bar(E_STFULL0 + ss));
                  bulk_load(st + 1024, a.rowds + int64_t(it) * a.Lpad + t * 128, 512, bar(E_STFULL0 + ss));
                  ++st_iss;
                  if (!(ok = mbar_wait(bar(E_QEMPTY), (sc & 1) ^ 1, abort_flag))) break;
                  mbar_expect_tx(bar(E_QFULL), 2 * C::kQBytes);
                  for (int hf = 0; hf < 4; ++hf)
                    for (int rh = 0; rh < 2; ++rh)
                      tma_load_5d(sbase + C::kOffQ0 + hf * 16384 + rh * C::kQBox, &tm_q, bar(E_QFULL), hf * 64, h,
                                  t * 128 + rh * QR, c, b);
                  ++q_iss;
                  if (!(ok = mbar_wait(bar(E_DOEMPTY), (sc & 1) ^ 1, abort_flag))) break;
                  mbar_expect_tx(bar(E_DOFULL), 2 * C::kQBytes);
                  for (int hf = 0; hf < 4; ++hf)
                    for (int rh = 0; rh < 2; ++rh)
                      tma_load_5d(sbase + C::kOffDO0 + hf * 16384 + rh * C::kQBox, &tm_do, bar(E_DOFULL), hf * 64, h,
                                  t * 128 + rh * QR, c, b);
                  ++do_iss;
                }
            }
          }
          if (!ok) break;
          // V into its place once pass 0's last S^T has read the Q tile there, and
          // pass 1's tiles once its last dV has read the dO tile
          if (!(ok = mbar_wait(bar(E_QEMPTY), (sc & 1) ^ 1, abort_flag))) break;
          mbar_expect_tx(bar(E_VFULL), C::kKVBytes);
          for (int hf = 0; hf < 4; ++hf)
            tma_load_5d(sV + hf * 16384, &tm_v, bar(E_VFULL), hf * 64, g, W[W_LROW], kc, kb);
          ++v_iss;
          if (!(ok = mbar_wait(bar(E_DOEMPTY), (sc & 1) ^ 1, abort_flag))) break;
          // pass 1: 64-row steps in reverse order
          const StepRange<QR> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
          for (int ii = 0; ii < R.it_hi - R.it_lo && ok; ++ii) {
            const int it = R.it_hi - 1 - ii;
            int t0, t1, r0;
            if (!R.tiles(it, t0, t1, r0)) continue;
            const int32_t* I = items + it * kItemWords;
            const int b = I[I_B], c = I[I_C];
            for (int tt = 0; tt <= t1 - t0 && ok; ++tt)
              for (int h2 = 0; h2 < a.G && ok; ++h2, ++sc) {
                const int t = t1 - tt, hh = a.G - 1 - h2;
                const int h = g * a.G + hh;
                // row statistics into their own two-stage ring
                const int ss = sc & 1;
                if (!(ok = mbar_wait(bar(E_STEMPTY0 + ss), ((sc >> 1) & 1) ^ 1, abort_flag))) break;
                mbar_expect_tx(bar(E_STFULL0 + ss), C::kStatBytes);
                const uint32_t st = sbase + C::kOffStat + ss * C::kStatBytes;
                const int64_t srow = (int64_t(it) * a.H + h) * a.Lpad + t * QR;
                bulk_load(st, a.lse2 + srow, QR * 4, bar(E_STFULL0 + ss));
                bulk_load(st + QR * 4, a.dstat + srow, QR * 4, bar(E_STFULL0 + ss));
                bulk_load(st + 2 * QR * 4, a.rowds + int64_t(it) * a.Lpad + t * QR, QR * 4, bar(E_STFULL0 + ss));
                ++st_iss;
                if (!(ok = mbar_wait(bar(E_QEMPTY), (sc & 1) ^ 1, abort_flag))) break;
                mbar_expect_tx(bar(E_QFULL), C::kQBytes);
                for (int hf = 0; hf < 4; ++hf)
                  tma_load_5d(sQ + hf * C::kQBox, &tm_q, bar(E_QFULL), hf * 64, h, t * QR, c, b);
                ++q_iss;
                if (!(ok = mbar_wait(bar(E_DOEMPTY), (sc & 1) ^ 1, abort_flag))) break;
                mbar_expect_tx(bar(E_DOFULL), C::kQBytes);
                for (int hf = 0; hf < 4; ++hf)
                  tma_load_5d(sDO + hf * C::kQBox, &tm_do, bar(E_DOFULL), hf * 64, h, t * QR, c, b);
                ++do_iss;
              }
          }
        }
        if (!ok) {
          // wait for copies already issued before the shared memory goes away
          if (u > 0) mbar_wait_drain(bar(E_KVFULL), (u - 1) & 1);
          if (v_iss > 0) mbar_wait_drain(bar(E_VFULL), (v_iss - 1) & 1);
          if (q_iss > 0) mbar_wait_drain(bar(E_QFULL), (q_iss - 1) & 1);
          if (do_iss > 0) mbar_wait_drain(bar(E_DOFULL), (do_iss - 1) & 1);
          for (uint32_t x = (st_iss > 2 ? st_iss - 2 : 0); x < st_iss; ++x)
            mbar_wait_drain(bar(E_STFULL0 + (x & 1)), (x >> 1) & 1);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(128, QR, false, false);   // S^T, dP^T: N = query rows
        constexpr uint32_t idAcc = idesc_bf16(128, 256, false, true);  // dV, dK: B MN-major, N = d
        constexpr uint32_t idDQ = idesc_bf16(128, QR, true, true);     // dQ^T halves: both MN-major
        constexpr uint32_t idS0 = idesc_bf16(128, 128, false, false);  // pass 0 S^T: N = 128 query rows
        const uint32_t dQ0_k = sdesc_lo(sbase + C::kOffQ0, 16), dDO0_mn = sdesc_lo(sbase + C::kOffDO0, 16384);
        const uint32_t dK_k = sdesc_lo(sK, 16), dV_k = sdesc_lo(sV, 16), dQ_k = sdesc_lo(sQ, 16);
        const uint32_t dDO_k = sdesc_lo(sDO, 16), dQ_mn = sdesc_lo(sQ, C::kQBox), dDO_mn = sdesc_lo(sDO, C::kQBox);
        const uint32_t dDS_k = sdesc_lo(sDS, 16), dDS_mn = sdesc_lo(sDS, 16384);
        const uint32_t dK0_mn = sdesc_lo(sK, 16384), dK1_mn = sdesc_lo(sK + 32768, 16384);  // K^T, d halves
        // K-major steps of 16 columns cross a 64-column box every 4 steps (K / V boxes
        // hold 128 rows, Q / dO boxes 64); MN-major steps advance 16 rows of 128 bytes
        auto kstep_kv = [](int kk) { return uint32_t(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
        auto kstep_q = [](int kk) { return uint32_t(((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4); };
        auto mnstep = [](int kk) { return uint32_t((kk * 2048) >> 4); };
        uint32_t u = 0, ua = 0, sc = 0, s0 = 0, s1 = 0;
        bool ok = true;
        for (uint32_t uk = 0; ok; ++uk) {
          const int w = unit_take(bar(E_UFULL), bar(E_UEMPTY), unit_ring, uk, abort_flag, true);
          if (w == -2) ok = false;
          if (w < 0) break;
          const int32_t* W = work + w * kBwdWords;
          const int nsteps = W[W_NQ];
          if (nsteps == 0) continue;
          if (!(ok = mbar_wait(bar(E_KVFULL), u & 1, abort_flag))) break;
          // ---- pass 0: 128-row steps; S^T of step p in TMEM columns 128 ((s0 + p) & 1);
          // the next step's S^T goes out before this step's dV, so that its P^T is
          // formed while dV runs
          int n0 = 0;
          {
            const StepRange<128> R0{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
            for (int it = R0.it_lo; it < R0.it_hi; ++it) {
              int t0, t1, r0;
              if (R0.tiles(it, t0, t1, r0)) n0 += (t1 - t0 + 1) * a.G;
            }
          }
          auto issue_s0 = [&](uint32_t step, uint32_t buf) {  // S^T = K Q^T, 128 queries
            if (!(ok = mbar_wait(bar(E_QFULL), step & 1, abort_flag))) return;
            // buffer 1 is pass 1's dQ^T place: the dQ warps must have read the last one
            if (buf && !(ok = mbar_wait(bar(E_DQEMPTY), (s1 & 1) ^ 1, abort_flag))) return;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ss_lo(tmem + C::kColS + buf * 128, dK_k + kstep_kv(kk), dQ0_k + kstep_kv(kk), idS0, kk > 0);
            // one barrier per buffer: the next step's S^T may complete before the P^T
            // warps wait for this one's, and a shared barrier would then have
            // advanced two phases
            tc_commit(bar(E_S0FULL0 + buf));
            tc_commit(bar(E_QEMPTY));  // pass 0 reads Q only here
          };
          issue_s0(sc, s0 & 1);
          for (int p = 0; p < n0 && ok; ++p, ++sc) {
            if (p + 1 < n0) {
              issue_s0(sc + 1, (s0 + 1) & 1);
              if (!ok) break;
            }
            if (!(ok = mbar_wait(bar(E_PREADY0 + (s0 & 1)), (s0 >> 1) & 1, abort_flag))) break;
            if (p == 0 && !(ok = mbar_wait(bar(E_ACCFREE), (ua & 1) ^ 1, abort_flag))) break;
            if (!(ok = mbar_wait(bar(E_DOFULL), sc & 1, abort_flag))) break;
            tc_fence_after();
            // dV += P^T dO: P^T of query half h packed in TMEM columns [64 h, 64 h + 32)
            // of the step's buffer; dO (128 rows) MN-major across four 16 KB boxes
            const uint32_t pb = tmem + C::kColS + (s0 & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_lo(tmem + C::kColAcc, pb + (kk >> 2) * 64 + (kk & 3) * 8, dDO0_mn + mnstep(kk), idAcc,
                        (p > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar(E_DOEMPTY));
            ++s0;
            if (p == n0 - 1) tc_commit(bar(E_ACCDONE));
          }
          ++ua;
          // ---- pass 1: 64-row steps (V loaded meanwhile into its place)
          auto issue_s = [&](uint32_t step) {  // S^T = K Q^T, 64 queries
            if (!(ok = mbar_wait(bar(E_QFULL), step & 1, abort_flag))) return;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) mma_ss_lo(tmem + C::kColS, dK_k + kstep_kv(kk), dQ_k + kstep_q(kk), idS, kk > 0);
            tc_commit(bar(E_SFULL));
          };
          if (ok) issue_s(sc);
          for (int s = 0; s < nsteps && ok; ++s, ++sc) {
            if (!(ok = mbar_wait(bar(E_DOFULL), sc & 1, abort_flag))) break;
            if (s == 0 && !(ok = mbar_wait(bar(E_VFULL), u & 1, abort_flag))) break;  // V fill of unit u
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ss_lo(tmem + C::kColDP, dV_k + kstep_kv(kk), dDO_k + kstep_q(kk), idS, kk > 0);
            tc_commit(bar(E_DPFULL));
            tc_commit(bar(E_DOEMPTY));  // pass 1 reads dO only here
            if (!(ok = mbar_wait(bar(E_DSREADY), s1 & 1, abort_flag))) break;
            if (s == 0 && !(ok = mbar_wait(bar(E_ACCFREE), (ua & 1) ^ 1, abort_flag))) break;
            tc_fence_after();
            // dK += dS^T Q (the last reader of the Q tile, which then reloads
            // while dQ^T runs)
#pragma unroll
            for (int kk = 0; kk < QR / 16; ++kk)
              mma_ss_lo(tmem + C::kColAcc, dDS_k + 2 * kk, dQ_mn + mnstep(kk), idAcc, (s > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar(E_QEMPTY));
            if (s == nsteps - 1) tc_commit(bar(E_ACCDONE));
            if (!(ok = mbar_wait(bar(E_DQEMPTY), (s1 & 1) ^ 1, abort_flag))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_lo(tmem + C::kColDQ, dK0_mn + mnstep(kk), dDS_mn + mnstep(kk), idDQ, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_lo(tmem + C::kColDQ + QR, dK1_mn + mnstep(kk), dDS_mn + mnstep(kk), idDQ, kk > 0);
            tc_commit(bar(E_DQFULL));
            tc_commit(bar(E_DSFREE));
            ++s1;
            if (s == nsteps - 1) tc_commit(bar(E_KVEMPTY));
            else issue_s(sc + 1);
          }
          ++ua;
          ++u;
        }
        if (!ok) {
          tc_commit(bar(E_DRAIN));
          mbar_wait_drain(bar(E_DRAIN), 0);
        }
      }
    }
  } else if (warp < 12) {
    regs_set<C::kRegsCompute, C::kRegsLaunch>();
    // ------------------------------------------------------------ P^T / dS^T
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int jl = quarter * 32 + lane;  // key row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t sc = 0, s0 = 0, s1 = 0;
    bool ok = true;
    // P of one 32-query chunk for key j (this lane): the S^T columns at TMEM column
    // `col`, the chunk's log2 LSE and document starts in shared memory, its first
    // global row ci0; full: the whole step is visible to key j. p gets P (masked),
    // pk the packed bf16 pairs, keep the dropout keep bits (bit e: query e)
    auto chunk_p = [&](uint32_t col, const float* c_lse, const int32_t* c_ds, int ci0, bool full, int j,
                       uint32_t hq, uint32_t bseq, int key0, float (&p)[32], uint32_t (&pk)[16], uint32_t& keep) {
      {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + col, r);
        tmem_ld_wait();
        reg_fence(r);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = ld_shared_f4(c_lse + 4 * e4);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) p[4 * e4 + k] = ex2(fmaf(__uint_as_float(r[4 * e4 + k]), a.scale_log2, -lv[k]));
        }
      }
      if (!full) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (!((j >= c_ds[e]) && (j <= ci0 + e))) p[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(p[2 * e], p[2 * e + 1]);
      keep = 0u;
      if constexpr (DROP) {
        // one Philox call per 2-query block (word 2 (i mod 2) + (j mod 2) of
        // counter (j/2, i/2, h, b))
        const int ibase = ci0;
        if ((ibase & 1) == 0 && (key0 & 1) == 0) {
          // keys 2m, 2m + 1 are lanes 2m, 2m + 1: each lane makes every other
          // call of the pair and hands its partner the two words it needs
          const uint32_t odd = lane & 1;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const uint4 rr = philox4x32_10(
                make_uint4(uint32_t(j) >> 1, uint32_t(ibase >> 1) + 2 * m + odd, hq, bseq), a.drop_k0, a.drop_k1);
            const uint32_t ev = uint32_t(rr.x >= a.drop_thresh) | (uint32_t(rr.z >= a.drop_thresh) << 1);
            const uint32_t od = uint32_t(rr.y >= a.drop_thresh) | (uint32_t(rr.w >= a.drop_thresh) << 1);
            const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? ev : od, 1);
            const uint32_t lo = odd ? got : ev, hi = odd ? od : got;  // query blocks 2m, 2m + 1
            keep |= (lo | (hi << 2)) << (4 * m);
          }
        } else if ((ibase & 1) == 0) {
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const uint4 rr = philox4x32_10(make_uint4(uint32_t(j) >> 1, uint32_t(ibase >> 1) + e2, hq, bseq),
                                           a.drop_k0, a.drop_k1);
            const uint32_t w0 = (j & 1) ? rr.y : rr.x, w1 = (j & 1) ? rr.w : rr.z;
            keep |= (uint32_t(w0 >= a.drop_thresh) << (2 * e2)) | (uint32_t(w1 >= a.drop_thresh) << (2 * e2 + 1));
          }
        } else {
#pragma unroll 4
          for (int e = 0; e < 32; ++e) {
            const int i = ibase + e;
            const uint4 rr =
                philox4x32_10(make_uint4(uint32_t(j) >> 1, uint32_t(i) >> 1, hq, bseq), a.drop_k0, a.drop_k1);
            const uint32_t wd = (i & 1) ? ((j & 1) ? rr.w : rr.z) : ((j & 1) ? rr.y : rr.x);
            keep |= uint32_t(wd >= a.drop_thresh) << e;
          }
        }
      }
    };
    for (uint32_t uk = 0; ok; ++uk) {
      const int w = unit_take(bar(E_UFULL), bar(E_UEMPTY), unit_ring, uk, abort_flag, false);
      if (w == -2) ok = false;
      if (w < 0) break;
      const int32_t* W = work + w * kBwdWords;
      if (W[W_NQ] == 0) continue;
      const int j = W[W_KEY0] + jl;  // global key row
      const int key0 = W[W_KEY0];
      // pass 0: 128-row steps; this warp's 64 queries [64 half, 64 half + 64) in two
      // chunks; P^T (dropped and rescaled under dropout) into the step's S^T buffer
      // (TMEM columns 128 (s0 & 1) ..), packed inside the half's own S^T columns:
      // chunk ch of half h at 64 h + 16 ch (over S^T the chunk has already read)
      {
        const StepRange<128> R0{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
        for (int it = R0.it_lo; it < R0.it_hi && ok; ++it) {
          int t0, t1, r0;
          if (!R0.tiles(it, t0, t1, r0)) continue;
          const uint32_t bseq = uint32_t(items[it * kItemWords + I_B]);
          for (int t = t0; t <= t1 && ok; ++t)
            for (int hh = 0; hh < a.G && ok; ++hh, ++sc, ++s0) {
              const int ss = sc & 1;
              const uint32_t hq = uint32_t(W[W_G] * a.G + hh);
              const int i0 = r0 + t * 128;
              const float* st_lse = reinterpret_cast<const float*>(smem + C::kOffDS + ss * C::kStat0Bytes);
              const int32_t* st_ds = reinterpret_cast<const int32_t*>(st_lse + 2 * 128);
              if (!(ok = mbar_wait(bar(E_STFULL0 + ss), (sc >> 1) & 1, abort_flag))) break;
              if (!(ok = mbar_wait(bar(E_S0FULL0 + (s0 & 1)), (s0 >> 1) & 1, abort_flag))) break;
              tc_fence_after();
              const bool full = (j <= i0) && (j >= st_ds[127]);
              const uint32_t buf = (s0 & 1) * 128;
#pragma unroll 1
              for (int ch = 0; ch < 2; ++ch) {
                const int ib = half * 64 + ch * 32;
                float p[32];
                uint32_t pk[16], keep;
                chunk_p(C::kColS + buf + ib, st_lse + ib, st_ds + ib, i0 + ib, full, j, hq, bseq, key0, p, pk, keep);
                if constexpr (DROP) {
                  uint32_t pd[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e)
                    pd[e] = pack_bf16(((keep >> (2 * e)) & 1) ? p[2 * e] * a.drop_scale : 0.f,
                                      ((keep >> (2 * e + 1)) & 1) ? p[2 * e + 1] * a.drop_scale : 0.f);
                  tmem_st16(tmem + lane_base + C::kColS + buf + half * 64 + ch * 16, pd);
                } else {
                  tmem_st16(tmem + lane_base + C::kColS + buf + half * 64 + ch * 16, pk);
                }
              }
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(bar(E_PREADY0 + (s0 & 1)));
              mbar_arrive(bar(E_STEMPTY0 + ss));
            }
        }
      }
      // pass 1: 64-row steps in reverse order; this warp's 32 queries of the step
      const StepRange<QR> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
      const int ib = half * 32;
      for (int ii = 0; ii < R.it_hi - R.it_lo && ok; ++ii) {
        const int it = R.it_hi - 1 - ii;
        int t0, t1, r0;
        if (!R.tiles(it, t0, t1, r0)) continue;
        const uint32_t bseq = uint32_t(items[it * kItemWords + I_B]);
        for (int tt = 0; tt <= t1 - t0 && ok; ++tt)
          for (int h2 = 0; h2 < a.G && ok; ++h2, ++sc) {
            const int t = t1 - tt, hh = a.G - 1 - h2;
            const int ss = sc & 1;
            const uint32_t hq = uint32_t(W[W_G] * a.G + hh);  // query head
            const int i0 = r0 + t * QR;                        // global row of query column 0
            const float* st_lse = reinterpret_cast<const float*>(smem + C::kOffStat + ss * C::kStatBytes);
            const float* st_d = st_lse + QR;
            const int32_t* st_ds = reinterpret_cast<const int32_t*>(st_lse + 2 * QR);
            if (!(ok = mbar_wait(bar(E_STFULL0 + ss), (sc >> 1) & 1, abort_flag))) break;
            if (!(ok = mbar_wait(bar(E_SFULL), s1 & 1, abort_flag))) break;  // pass-1 S^T number s1
            tc_fence_after();
            // rows' document starts are non-decreasing and invalid rows carry INT_MAX,
            // so key j sees every query of the step iff it lies at or before the
            // step's first row and at or after the last row's document start
            const bool full = (j <= i0) && (j >= st_ds[QR - 1]);
            uint32_t pk[16];
            float p[32];
            uint32_t keep;  // dropout: bit e keeps query i0 + ib + e for this key
            chunk_p(C::kColS + ib, st_lse + ib, st_ds + ib, i0 + ib, full, j, hq, bseq, key0, p, pk, keep);
            if (!(ok = mbar_wait(bar(E_DPFULL), s1 & 1, abort_flag))) break;
            tc_fence_after();
            uint32_t dsk[16];
            {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + C::kColDP + ib, r);
              tmem_ld_wait();
              reg_fence(r);
#pragma unroll
              for (int e4 = 0; e4 < 8; ++e4) {
                const float4 d4 = ld_shared_f4(st_d + ib + 4 * e4);
                const int e = 4 * e4;
                const uint32_t p01 = pk[2 * e4], p23 = pk[2 * e4 + 1];
                float dp[4] = {__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                               __uint_as_float(r[e + 3])};
                if constexpr (DROP) {
                  // dS = P (keep dP / (1 - p) - D) with the undropped P
#pragma unroll
                  for (int k = 0; k < 4; ++k) dp[k] = ((keep >> (e + k)) & 1) ? dp[k] * a.drop_scale : 0.f;
                }
                dsk[2 * e4] = pack_bf16(__uint_as_float(p01 << 16) * (dp[0] - d4.x),
                                        __uint_as_float(p01 & 0xffff0000u) * (dp[1] - d4.y));
                dsk[2 * e4 + 1] = pack_bf16(__uint_as_float(p23 << 16) * (dp[2] - d4.z),
                                            __uint_as_float(p23 & 0xffff0000u) * (dp[3] - d4.w));
              }
            }
            mbar_arrive(bar(E_STEMPTY0 + ss));
            // dS^T of the previous pass-1 step must have been read by its dK and dQ^T
            if (s1 > 0 && !(ok = mbar_wait(bar(E_DSFREE), (s1 - 1) & 1, abort_flag))) break;
            // dS^T rows: 64 queries = one 128-byte row per key (128-byte swizzle); this
            // warp's 32 queries are its 16-byte pieces 4 half .. 4 half + 3
            const uint32_t row_addr = sDS + jl * 128;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
              st_shared_v4(row_addr + (((half * 4 + c4) ^ (jl & 7)) << 4), dsk[4 * c4], dsk[4 * c4 + 1],
                           dsk[4 * c4 + 2], dsk[4 * c4 + 3]);
            fence_proxy_async_smem();
            mbar_arrive(bar(E_DSREADY));
            ++s1;
          }
      }
    }
  } else {
    regs_set<C::kRegsDq, C::kRegsLaunch>();
    // ------------------------------------------------------------ dQ out, dV / dK epilogue
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // TMEM lane: column of dQ^T within a d half, key row of dV / dK
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t ua = 0, s1 = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      const int w = unit_take(bar(E_UFULL), bar(E_UEMPTY), unit_ring, uk, abort_flag, false);
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
          for (int k = 0; k < 64; ++k) {
            reinterpret_cast<float4*>(dkrow)[k] = z;
            reinterpret_cast<float4*>(dvrow)[k] = z;
          }
        }
        continue;
      }
      const StepRange<QR> R{items, W[W_ITEM_LO], W[W_ITEM_HI], W[W_QLO], W[W_QHI], a.L};
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          for (int ii = 0; ii < R.it_hi - R.it_lo && ok; ++ii) {
            const int it = R.it_hi - 1 - ii;
            int t0, t1, r0;
            if (!R.tiles(it, t0, t1, r0)) continue;
            const int32_t* I = items + it * kItemWords;
            const int b = I[I_B], c = I[I_C];
            for (int tt = 0; tt <= t1 - t0 && ok; ++tt)
              for (int h2 = 0; h2 < a.G && ok; ++h2, ++s1) {
                const int t = t1 - tt, hh = a.G - 1 - h2;
                const int h = g * a.G + hh;
                // the four dQ warps leave together (they meet at named barriers below)
                ok = bar_red_and(1, 128, mbar_wait(bar(E_DQFULL), s1 & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                // r[2 dh + k]: column 128 dh + rl of dQ^T, query rows 32 k .. 32 k + 31
                uint32_t r[4][32];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(tmem + lane_base + C::kColDQ + q * 32, r[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) reg_fence(r[q]);
                tc_fence_before();
                mbar_arrive(bar(E_DQEMPTY));
                // 16-row x 128-column boxes (one d half, 8 KB, row-major, unswizzled:
                // each warp writes its 32 columns of a row as one 128-byte run) built
                // by the four warps together in two buffers, each sent with one TMA
                // reduce-add (rows past L are clipped). An SM's reduce-adds proceed one
                // box at a time at about the same cost up to 8 KB, so four warps
                // sending 2 KB boxes of 32 columns took four times as long.
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int dh = k >> 2, rr = k & 3;
                  const uint32_t buf = sStage + (k & 1) * 8192;
                  if (rl == 0) bulk_wait_read<1>();  // the box sent from this buffer two rounds ago has left it
                  named_bar_sync(1, 128);
#pragma unroll
                  for (int q = 0; q < 16; ++q) {
                    const int row = rr * 16 + q;
                    st_shared_f32(buf + q * 512 + rl * 4, __uint_as_float(r[2 * dh + (row >> 5)][row & 31]) * a.scale);
                  }
                  fence_proxy_async_smem();
                  named_bar_sync(1, 128);
                  if (rl == 0) {
                    tma_reduce_add_5d(&tm_dq, buf, dh * 128, h, t * QR + rr * 16, c, b);
                    bulk_commit();
                  }
                }
              }
          }
          if (!ok) break;
        }
        if (!(ok = mbar_wait(bar(E_ACCDONE), ua & 1, abort_flag))) break;
        tc_fence_after();
        // dV (pass 0) or dK x scale (pass 1), in two 128-column halves; the
        // accumulator is released once both have left TMEM
        float* row = pass ? dkrow : dvrow;
        const float mul = pass ? a.scale : 1.f;
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {
          uint32_t v[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tmem + lane_base + C::kColAcc + x * 128 + q * 32, v[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) reg_fence(v[q]);
          if (x == 1) {
            tc_fence_before();
            mbar_arrive(bar(E_ACCFREE));
          }
          if (krow_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float4 o = make_float4(__uint_as_float(v[q][4 * e]) * mul, __uint_as_float(v[q][4 * e + 1]) * mul,
                                       __uint_as_float(v[q][4 * e + 2]) * mul, __uint_as_float(v[q][4 * e + 3]) * mul);
                float4* pp = reinterpret_cast<float4*>(row + x * 128 + q * 32) + e;
                if (a.accumulate) {
                  const float4 old = *pp;
                  o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                }
                *pp = o;
              }
          }
        }
        ++ua;
      }
      if (!ok) break;
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

template <bool DROP>
int32_t launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                   const CUtensorMap& mdq, const BwdArgs& a, int grid, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(bd_bwd256_kernel<DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg256::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd256)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, bd_bwd256_kernel<DROP>);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(bwd256)");
    // the setmaxnreg directions were chosen for this launch count: refuse any other
    if (fa.numRegs != Cfg256::kRegsLaunch)
      return fail(BD_ERR_UNSUPPORTED, "bwd256 kernel built with %d registers/thread, its register split assumes %d",
                  fa.numRegs, Cfg256::kRegsLaunch);
    attr_done[dev] = true;
  }
  bd_bwd256_kernel<DROP><<<grid, Cfg256::kThreads, Cfg256::kSmem, stream>>>(mq, mk, mv, mdo, mdq, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bd_bwd256_kernel launch");
  return BD_OK;
}

}  // namespace

int32_t launch_bwd256(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                      const CUtensorMap& mdq, const BwdArgs& a, bool drop, int grid, cudaStream_t stream) {
  return drop ? launch_one<true>(mq, mk, mv, mdo, mdq, a, grid, stream)
              : launch_one<false>(mq, mk, mv, mdo, mdq, a, grid, stream);
}

}  // namespace bd
