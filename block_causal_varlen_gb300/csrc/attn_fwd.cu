// Forward of block-causal varlen chunked attention on sm_103a.
//
// What it computes (NeMo Automodel page "block-diagonal varlen CP for packed
// sequences", Summary and Key correctness properties 1-2): for every query row
// i of a chunk, O_i = softmax_j(scale * q_i . k_j) v_j over the keys j of row
// i's own document with j <= i, plus LSE_i (natural log, fp32). Rows past the
// valid length give O = 0 and LSE = -inf.
//
// Design (one persistent CTA per SM, 12 warps; each CTA claims its next work
// unit from a per-launch counter when it is ready for it, so the units, listed
// longest first, spread evenly however long each one is):
//   warp 0      TMA producer: Q tiles of the two query heads, then a ring of
//               K/V tiles (128 keys x d) for the work unit's key-tile range
//               [kt_lo, kt_lo + nt); fully masked tiles are never loaded.
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma.
//   warps 4-7   softmax for query head h0   (slot 0, TMEM lanes = rows)
//   warps 8-11  softmax for query head h0+1 (slot 1), same rows and keys
// The two slots are two query heads of one GQA group, so each K/V tile in
// shared memory feeds both; while one slot's softmax runs, the tensor core
// works on the other slot (S = Q K^T into TMEM, then O += P V with P read
// straight from TMEM). TMEM columns: S0 [0,128), S1 [128,256), O0 and O1
// after that; P_s (bf16 pairs) overwrites the first 64 columns of S_s.
// Online softmax works in the log2 domain and only rescales O when the row
// maximum grows by more than 2^8 (exact: the final 1/l uses the same stale max).
// Head dim 256 runs one slot per CTA (its O takes TMEM columns 256..511).
// The DROP instantiation applies attention dropout to P before the PV product
// with a Philox4x32-10 keep mask (Salmon et al., SC 2011) regenerated from the
// plan's seed; the row sum keeps the undropped values and 1/(1-p) is applied
// with 1/l in the epilogue.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <math_constants.h>

#include <atomic>
#include <cstring>

#include "host_util.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace bd {
using namespace dev;

struct FwdArgs {
  const int32_t* plan;
  __nv_bfloat16* o;
  int64_t o_sb, o_sc, o_sr, o_sh;
  float* lse;
  int64_t l_sb, l_sc, l_sh;
  int32_t L, n_work, slots, Ck;
  float scale_log2;
  // attention dropout (used by the DROP instantiation): keep iff Philox word >= thresh
  uint32_t drop_thresh, drop_k0, drop_k1;
  float drop_scale;
  // optional fp32 tensor [B, C, L, H, d] (the backward's dQ accumulator) that the
  // otherwise idle warps 2-3 set to zero while the forward runs; NULL for none
  float* dqz;
  int64_t z_sb, z_sc, z_sr, z_sh;
  int32_t B, C, H;
  int32_t counter_slot;  // which (claim, done) pair of the plan's forward counter slots
};

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // 128 rows x D bf16
  // K and V have rings of their own: a K tile is released as soon as both
  // slots' S MMAs have read it, so it can be refilled well ahead of its use.
  // head dim 256: one query-head slot (its O takes TMEM columns 256..511) and
  // single 64 KB K and V stages
  static constexpr int kQSlots = (D == 256) ? 1 : 2;
  static constexpr int kKStages = (D == 256) ? 1 : (D == 128) ? 2 : 4;
  static constexpr int kVStages = (D == 256) ? 1 : (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  // head dims 64 / 128: one 16 KB staging box (128 rows x 64 columns bf16) per slot
  // through which the epilogue's O rows leave by TMA
  static constexpr int kStageBytes = 16384;
  static constexpr int kOffStage = kOffV + kVStages * kTileBytes;
  static constexpr int kOffBar = kOffStage + (D <= 128 ? 2 * kStageBytes : 0);
  // the 128 rows' document starts of a unit's query tile, two buffers (units in turn)
  static constexpr int kOffDs = kOffBar + 512;
  static constexpr int kSmem = kOffDs + 2 * 512 + 1024;  // + alignment slack
  static constexpr int kOCol = 256;                   // first O column in TMEM
  static constexpr int kThreads = 384;
  // register split after setmaxnreg: warpgroup 0 (producer, MMA) and the two
  // softmax warpgroups; the sum must fit in what the launch reserved
  static constexpr int kRegsCtl = 72, kRegsSoftmax = 216;
  static constexpr int kRegsNeeded = 128 * kRegsCtl + 256 * kRegsSoftmax;
  static constexpr int kRegsLaunch = 168;  // 65536 / 384 threads, rounded down to 8
  static_assert(kRegsNeeded <= kRegsLaunch * kThreads, "register split exceeds the launch's registers");
  static_assert(kSmem <= 232448, "shared memory over the per-CTA limit");
  static_assert(kOCol + kQSlots * D <= 512, "O accumulators exceed TMEM");
};

// barrier indices (8 bytes each)
enum : int {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = 6, B_VFULL = 10, B_VEMPTY = 14, B_SFULL = 18,
  B_PFULL = 20, B_OFINAL = 22, B_OEMPTY = 24, B_DRAIN = 26, B_TURN = 28, B_DSFULL = 30, B_UFULL = 32,
  B_UEMPTY = 32 + kUnitSlots, B_COUNT = 32 + 2 * kUnitSlots
};
// Each slot of the forward's unit ring carries, besides the unit index, the unit's
// words that the MMA and softmax warps need. The producer, which runs ahead of
// them, reads these from global memory (a dependent chain: the unit, then its
// item), so that a unit's first tile does not wait on those loads.
enum : int { R_W = 0, R_NT, R_ITEM, R_QTILE, R_H0, R_KTLO, R_B, R_C, R_ROW0, kRingWords = 10 };
static_assert(8 * B_COUNT + 16 + 4 * kUnitSlots * kRingWords <= 512,
              "barriers, TMEM slot, abort flag and unit ring overflow their region");

struct FwdUnit {
  int w, nt, item, qtile, h0, ktlo, b, c, row0;
};

// Consumer side of ring entry k: every lane of a warp (or a lone thread with
// one_thread set) copies the entry; one arrival per warp releases it. u.w is the
// unit (-1: no more work, -2: the wait gave up).
__device__ __forceinline__ void fwd_unit_take(uint32_t full0, uint32_t empty0, const volatile int32_t* ring,
                                              uint32_t k, volatile int* abort, bool one_thread, FwdUnit& u) {
  const int s = int(k % kUnitSlots);
  const bool ok = mbar_wait(full0 + 8u * s, (k / kUnitSlots) & 1, abort);
  const volatile int32_t* R = ring + s * kRingWords;
  u.w = ok ? R[R_W] : -2;
  if (u.w >= 0) {
    u.nt = R[R_NT]; u.item = R[R_ITEM]; u.qtile = R[R_QTILE]; u.h0 = R[R_H0]; u.ktlo = R[R_KTLO];
    u.b = R[R_B]; u.c = R[R_C]; u.row0 = R[R_ROW0];
  }
  if (!one_thread) __syncwarp();
  if (ok && (one_thread || (threadIdx.x & 31) == 0)) mbar_arrive(empty0 + 8u * s);
}

template <int D, bool DROP>
__global__ void __launch_bounds__(384, 1)
    bd_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdArgs a) {
  using Cfg = FwdCfg<D>;
  constexpr int NK = Cfg::kKStages, NV = Cfg::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + Cfg::kOffQ, sK = sbase + Cfg::kOffK, sV = sbase + Cfg::kOffV;
  const uint32_t sDs = sbase + Cfg::kOffDs;
  const uint32_t bars = sbase + Cfg::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffBar + 8 * B_COUNT + 8);
  volatile int32_t* unit_ring = reinterpret_cast<volatile int32_t*>(smem + Cfg::kOffBar + 8 * B_COUNT + 16);
  int* claim = const_cast<int32_t*>(a.plan) + H_FWD_SLOTS + 2 * a.counter_slot;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t* plan = a.plan;
  const int32_t* work = plan + plan[H_OFF_FWD];
  const int32_t* items = plan + plan[H_OFF_ITEMS];
  const int32_t* rowds_all = plan + plan[H_OFF_ROWDS];  // [nitems][Lpad]
  const int Lpad = plan[H_QTILES] * 128;
  const int slots = a.slots;

  if (threadIdx.x == 0) {
    // each slot's MMA thread releases the shared Q / K / V stages: one arrival per slot
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), slots);
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), slots);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), slots);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_DSFULL + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), 128);
      mbar_init(bar(B_OFINAL + s), 1);
      mbar_init(bar(B_OEMPTY + s), 128);
      mbar_init(bar(B_DRAIN + s), 1);
      mbar_init(bar(B_TURN + s), 1);
    }
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(bar(B_UFULL + s), 1);
      mbar_init(bar(B_UEMPTY + s), 5 * slots);  // each slot's MMA thread and softmax warps
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
  // the softmax warpgroups hold a 128-column score row each: registers move to
  // them from warpgroup 0 (producer and MMA warps) at the top of each branch
  if (warp < 4) {
   regs_set<Cfg::kRegsCtl, Cfg::kRegsLaunch>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t k_it = 0, v_it = 0, qi = 0;
      bool ok = true;
      const int G = plan[H_G];
      for (uint32_t uk = 0; ok; ++uk) {
        // claim the next unit and publish it with its words
        const int us = int(uk % kUnitSlots);
        if (!(ok = mbar_wait(bar(B_UEMPTY + us), ((uk / kUnitSlots) & 1) ^ 1, abort_flag))) break;
        int w = atomicAdd(claim, 1);
        if (w >= a.n_work) w = -1;
        volatile int32_t* R = unit_ring + us * kRingWords;
        int nt = 0, h0 = 0, qtile = 0, ktlo = 0, b = 0, c = 0, kvbuf = 0, kvbase = 0, item = 0;
        if (w >= 0) {
          const int32_t* W = work + w * kFwdWords;
          item = W[F_ITEM];
          nt = W[F_NT]; h0 = W[F_H0]; qtile = W[F_QTILE]; ktlo = W[F_KTLO];
          const int32_t* I = items + item * kItemWords;
          b = I[I_B]; c = I[I_C]; kvbuf = I[I_KVBUF]; kvbase = I[I_KVBASE];
          R[R_NT] = nt; R[R_ITEM] = item; R[R_QTILE] = qtile; R[R_H0] = h0; R[R_KTLO] = ktlo;
          R[R_B] = b; R[R_C] = c; R[R_ROW0] = I[I_ROW0];
        }
        R[R_W] = w;
        mbar_arrive(bar(B_UFULL + us));
        if (w < 0) break;
        if (nt == 0) continue;
        const int g = h0 / G;
        const int kb = kvbuf / a.Ck, kc = kvbuf % a.Ck;
        if (!(ok = mbar_wait(bar(B_QEMPTY), (qi & 1) ^ 1, abort_flag))) break;
        mbar_expect_tx(bar(B_QFULL), slots * Cfg::kTileBytes);
        for (int s = 0; s < slots; ++s)
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_5d(sQ + s * Cfg::kTileBytes + hf * 16384, &tm_q, bar(B_QFULL), hf * 64, h0 + s,
                        qtile * 128, c, b);
        // the tile rows' document starts for the softmax warps (buffer qi & 1 was
        // last read at the start of unit qi - 2, before that unit's first P and so
        // before the S that released the Q stage just waited for)
        mbar_expect_tx(bar(B_DSFULL + (qi & 1)), 512);
        bulk_load(sDs + (qi & 1) * 512, rowds_all + int64_t(item) * Lpad + qtile * 128, 512, bar(B_DSFULL + (qi & 1)));
        ++qi;
        for (int j = 0; j < nt; ++j) {
          const int row = (ktlo + j) * 128 - kvbase;
          const int sk = k_it % NK, sv = v_it % NV;
          BD_TRACE_EVENT(24, int(k_it));  // producer: waits for a K stage
          if (!(ok = mbar_wait(bar(B_KEMPTY + sk), ((k_it / NK) & 1) ^ 1, abort_flag))) break;
          BD_TRACE_EVENT(23, int(k_it));  // producer: K load issued
          mbar_expect_tx(bar(B_KFULL + sk), Cfg::kTileBytes);
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_5d(sK + sk * Cfg::kTileBytes + hf * 16384, &tm_k, bar(B_KFULL + sk), hf * 64, g, row, kc,
                        kb);
          ++k_it;
          BD_TRACE_EVENT(25, int(v_it));  // producer: waits for a V stage
          if (!(ok = mbar_wait(bar(B_VEMPTY + sv), ((v_it / NV) & 1) ^ 1, abort_flag))) break;
          BD_TRACE_EVENT(22, int(v_it));  // producer: V load issued
          mbar_expect_tx(bar(B_VFULL + sv), Cfg::kTileBytes);
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_5d(sV + sv * Cfg::kTileBytes + hf * 16384, &tm_v, bar(B_VFULL + sv), hf * 64, g, row, kc,
                        kb);
          ++v_it;
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA's shared memory goes away
        for (int s = 0; s < NK; ++s)
          if (k_it > uint32_t(s)) {
            const uint32_t last = k_it - 1 - ((k_it - 1 - s) % NK);
            mbar_wait_drain(bar(B_KFULL + s), (last / NK) & 1);
          }
        for (int s = 0; s < NV; ++s)
          if (v_it > uint32_t(s)) {
            const uint32_t last = v_it - 1 - ((v_it - 1 - s) % NV);
            mbar_wait_drain(bar(B_VFULL + s), (last / NV) & 1);
          }
        if (qi > 0) mbar_wait_drain(bar(B_QFULL), (qi - 1) & 1);
        for (uint32_t x = (qi > 2 ? qi - 2 : 0); x < qi; ++x) mbar_wait_drain(bar(B_DSFULL + (x & 1)), (x >> 1) & 1);
      }
    }
  } else if (warp == 1 || (warp == 2 && slots == 2)) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per query-head slot (warp 1: slot 0, warp 2: slot 1) issues that
    // slot's S = Q K^T and O += P V. An MMA issue only returns once the tensor pipe
    // has taken the previous one, so a single issuer leaves the pipe idle while it
    // commits or checks a barrier. The two issuers take turns group by group (a
    // group: a slot's PV then its next S), which keeps the slots' softmaxes
    // staggered as with one issuer, while each one's commits and barrier checks
    // overlap the other's issue. B_TURN + s completes when slot s may issue its
    // next group.
    if (lane == 0) {
      const int s = warp - 1;
      const bool turns = slots == 2;
      uint32_t my_turn = 0;  // groups this slot has issued
      // waits for this slot's turn (slot 0 goes first) and, after the group,
      // hands the turn to the other slot
      auto take_turn = [&]() -> bool {
        if (!turns || (s == 0 && my_turn == 0)) return true;
        const uint32_t k = s == 0 ? my_turn - 1 : my_turn;  // the other slot's groups done before mine
        return mbar_wait_spin(bar(B_TURN + s), k & 1, abort_flag);
      };
      auto pass_turn = [&]() {
        if (turns) mbar_arrive(bar(B_TURN + (s ^ 1)));
        ++my_turn;
      };
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      const uint32_t d_s = tmem + s * 128, d_o = tmem + Cfg::kOCol + s * D;
      const uint32_t qa = sdesc_lo(sQ + s * Cfg::kTileBytes, 16);
      // descriptors are built once per operand tile; a K step only advances the
      // start-address field (16-byte units) with a 64-bit add
      auto issue_s = [&](int st) {
        const uint32_t kb = sdesc_lo(sK + st * Cfg::kTileBytes, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = uint32_t(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_ss_lo(d_s, qa + off, kb + off, idS, kk > 0);
        }
      };
      auto issue_pv = [&](int st, bool acc) {
        const uint32_t vb = sdesc_lo(sV + st * Cfg::kTileBytes, 16384);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts_lo(d_o, d_s + kk * 8, vb + uint32_t(kk * 128), idPV, (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t kv_it = 0, qi = 0, tcount = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        FwdUnit U;
        fwd_unit_take(bar(B_UFULL), bar(B_UEMPTY), unit_ring, uk, abort_flag, true, U);
        if (U.w == -2) ok = false;
        if (U.w < 0) break;
        const int nt = U.nt;
        if (nt == 0) continue;
        if (!(ok = mbar_wait(bar(B_QFULL), qi & 1, abort_flag))) break;
        {
          const int sk0 = kv_it % NK;
          if (!(ok = mbar_wait(bar(B_KFULL + sk0), (kv_it / NK) & 1, abort_flag))) break;
          if (!(ok = take_turn())) break;
          tc_fence_after();
          issue_s(sk0);
          pass_turn();
          tc_commit(bar(B_SFULL + s));
          tc_commit(bar(B_KEMPTY + sk0));
          if (nt == 1) tc_commit(bar(B_QEMPTY));
        }
        for (int j = 1; j <= nt && ok; ++j) {
          const uint32_t itp = kv_it + j - 1, itn = kv_it + j;
          const int svp = itp % NV, skn = itn % NK;
          const uint32_t tp = tcount + j - 1;
          BD_TRACE_EVENT(14 + s, int(tp));  // MMA: starts waiting for P
          if (!(ok = mbar_wait_spin(bar(B_PFULL + s), tp & 1, abort_flag))) break;
          if (j == 1 && !(ok = mbar_wait(bar(B_OEMPTY + s), (qi & 1) ^ 1, abort_flag))) break;
          if (!(ok = mbar_wait(bar(B_VFULL + svp), (itp / NV) & 1, abort_flag))) break;
          if (j < nt && !(ok = mbar_wait(bar(B_KFULL + skn), (itn / NK) & 1, abort_flag))) break;
          if (!(ok = take_turn())) break;
          tc_fence_after();
          BD_TRACE_EVENT(10 + s, int(tp));  // MMA: P ready, PV issued
          issue_pv(svp, j > 1);
          if (j < nt) issue_s(skn);
          pass_turn();
          tc_commit(bar(B_VEMPTY + svp));
          if (j < nt) {
            BD_TRACE_EVENT(12 + s, int(tcount + j));  // MMA: S issued
            tc_commit(bar(B_SFULL + s));
            tc_commit(bar(B_KEMPTY + skn));
            if (j == nt - 1) tc_commit(bar(B_QEMPTY));
          } else {
            tc_commit(bar(B_OFINAL + s));
          }
        }
        kv_it += nt;
        tcount += nt;
        ++qi;
      }
      if (!ok) {
        tc_commit(bar(B_DRAIN + s));
        mbar_wait_drain(bar(B_DRAIN + s), 0);
      }
    }
   }
   else if (warp == 3) {
    // warp 3: zero the caller's dQ accumulator, one (row, head) d-vector per warp
    // store round, rows spread over every CTA of the launch (32-bit index
    // arithmetic once per row)
    if (a.dqz != nullptr) {
      const int rows = a.B * a.C * a.L;
      for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const int l = row % a.L, bc = row / a.L;
        float* p = a.dqz + int64_t(bc / a.C) * a.z_sb + int64_t(bc % a.C) * a.z_sc + int64_t(l) * a.z_sr;
        for (int h = 0; h < a.H; ++h)
#pragma unroll
          for (int col = lane * 4; col < D; col += 128)
            *reinterpret_cast<float4*>(p + int64_t(h) * a.z_sh + col) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#ifdef BD_TRACE
    if (lane == 0 && blockIdx.x == 0) {
      // tracing build only: stamp the moment each K tile lands
      for (uint32_t it = 0; it < uint32_t(kTraceTiles); ++it) {
        const uint32_t fb = bar(B_KFULL + int(it % NK)), par = (it / NK) & 1;
        const uint64_t t0 = globaltimer();
        bool got = false;
        while (!(got = mbar_try_wait(fb, par)) && globaltimer() - t0 < 20000000ull) {
        }
        if (!got) break;
        BD_TRACE_EVENT(26, int(it));
      }
    }
#endif
   }
  } else {
    regs_set<Cfg::kRegsSoftmax, Cfg::kRegsLaunch>();
    // ------------------------------------------------------------ softmax
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + s * 128;
    const uint32_t tO = tmem + lane_base + Cfg::kOCol + s * D;
    if (s < slots) {
      uint32_t tcount = 0, qi = 0;
      bool ok = true;
      // the next unit is taken from the ring before this unit's epilogue
      FwdUnit U;
      auto take = [&](uint32_t k, FwdUnit& X) {
        fwd_unit_take(bar(B_UFULL), bar(B_UEMPTY), unit_ring, k, abort_flag, false, X);
      };
      const int32_t* ds_buf = reinterpret_cast<const int32_t*>(smem + Cfg::kOffDs);
      take(0, U);
      for (uint32_t uk = 0; ok; ++uk) {
        if (U.w == -2) ok = false;
        if (U.w < 0) break;
        const int nt = U.nt;
        const int b = U.b, c = U.c;
        const int h = U.h0 + s;
        const int lrow = U.qtile * 128 + r;  // row within the chunk
        const int grow = U.row0 + lrow;      // global row
        const bool row_ok = lrow < a.L;
        // the row's document start, loaded with the unit's Q tile (rows past L are
        // invalid); not needed by a unit without tiles
        int ds = kRowInvalid;
        if (nt > 0) {
          if (!(ok = mbar_wait(bar(B_DSFULL + (qi & 1)), (qi >> 1) & 1, abort_flag))) break;
          ds = ds_buf[(qi & 1) * 128 + r];
        }
        const bool valid = ds != kRowInvalid;
        (void)grow;
        __nv_bfloat16* orow = a.o + b * a.o_sb + c * a.o_sc + int64_t(lrow) * a.o_sr + int64_t(h) * a.o_sh;
        float* lrow_p = a.lse + b * a.l_sb + c * a.l_sc + int64_t(h) * a.l_sh + lrow;
        if (nt == 0) {
          if (row_ok) {
            uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < D / 8; ++k) reinterpret_cast<uint4*>(orow)[k] = z;
            *lrow_p = -CUDART_INF_F;
          }
          take(uk + 1, U);
          continue;
        }
        float m_run = -CUDART_INF_F, l_run = 0.f;
        for (int j = 0; j < nt; ++j, ++tcount) {
          if (r == 0) BD_TRACE_EVENT(20 + s, int(tcount));  // softmax: start waiting for S
          if (!(ok = mbar_wait(bar(B_SFULL + s), tcount & 1, abort_flag))) break;
          tc_fence_after();
          if (r == 0) BD_TRACE_EVENT(30 + s, int(tcount));  // softmax: S ready
          uint32_t u[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, u[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) reg_fence(u[q]);
          float x[128];
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e) x[q * 32 + e] = __uint_as_float(u[q][e]);
          // the row sees the tile's columns [lo, hi] (none when the row is invalid)
          const int c0 = (U.ktlo + j) * 128;
          const int lo = valid ? ds - c0 : 128, hi = valid ? grow - c0 : -1;
          // Per 32-column group, for the whole warp: bit q of `gone` is set when no row
          // sees any column of group q (cleared without tests, left out of the row
          // max); groups every row sees whole are left alone; only the others are
          // masked element by element.
          uint32_t gone = 0;
          if (__any_sync(0xffffffffu, !(lo <= 0 && hi >= 127))) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (__all_sync(0xffffffffu, hi < 32 * q || lo > 32 * q + 31)) {
                gone |= 1u << q;
#pragma unroll
                for (int e = 0; e < 32; ++e) x[32 * q + e] = -CUDART_INF_F;
              } else if (!__all_sync(0xffffffffu, lo <= 32 * q && hi >= 32 * q + 31)) {
                // bit e of `seen`: the row sees column 32 q + e (one bit test per element)
                const int a0 = lo - 32 * q, a1 = hi - 32 * q;
                uint32_t seen = 0u;
                if (a1 >= 0 && a0 <= 31 && a1 >= a0)
                  seen = (a0 <= 0 ? 0xffffffffu : (0xffffffffu << a0)) & (a1 >= 31 ? 0xffffffffu : (0xffffffffu >> (31 - a1)));
#pragma unroll
                for (int e = 0; e < 32; ++e) x[32 * q + e] = (seen & (1u << e)) ? x[32 * q + e] : -CUDART_INF_F;
              }
            }
          }
          // row max: eight independent 3-input max chains, then a small tree
          float m8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = -CUDART_INF_F;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (!(gone & (1u << q)))
#pragma unroll
              for (int e = 32 * q; e < 32 * q + 32; e += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = max3f(m8[k], x[e + k], x[e + 8 + k]);
          const float mx = fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(max3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
          if (r == 0) BD_TRACE_EVENT(40 + s, int(tcount));  // softmax: row max done
          const float m_new = fmaxf(m_run, mx * a.scale_log2);
          const bool need = m_new > m_run + 8.0f;
          float factor = 1.f;
          if (need) {
            factor = ex2(m_run - m_new);
            l_run *= factor;
            m_run = m_new;
          }
          if (__any_sync(0xffffffffu, need && j > 0)) {
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
              uint32_t ov[32];
              tmem_ld32(tO + q * 32, ov);
              tmem_ld_wait();
              reg_fence(ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
              tmem_st32(tO + q * 32, ov);
            }
          }
          const float m_eff = (m_run == -CUDART_INF_F) ? 0.f : m_run;
          // p = 2^(x * scale_log2 - m): paired FMAs, then the exponentials; the
          // row sum uses four paired accumulators
          const float2 cs = make_float2(a.scale_log2, a.scale_log2), cm = make_float2(-m_eff, -m_eff);
          float2 s4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
          // dropout keep bits of the tile's 128 keys for this row, bit k of word k / 32
          // (keys c0 + 2e, c0 + 2e + 1 form one 2-key block: c0 is a multiple of 128)
          uint32_t kbits[4] = {0u, 0u, 0u, 0u};
          if constexpr (DROP) {
            const uint32_t T = a.drop_thresh, kb0 = uint32_t(c0) >> 1, rb = uint32_t(grow) >> 1;
            if ((U.row0 & 1) == 0) {
              // rows 2m, 2m + 1 are lanes 2m, 2m + 1: each lane makes every other call
              // of the pair and hands its partner the two words the partner needs
              const uint32_t odd = lane & 1;
#pragma unroll 8
              for (int m = 0; m < 32; ++m) {
                const uint4 rr = philox4x32_10(make_uint4(kb0 + 2 * m + odd, rb, uint32_t(h), uint32_t(b)),
                                               a.drop_k0, a.drop_k1);
                const uint32_t ev = uint32_t(rr.x >= T) | (uint32_t(rr.y >= T) << 1);
                const uint32_t od = uint32_t(rr.z >= T) | (uint32_t(rr.w >= T) << 1);
                const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? ev : od, 1);
                const uint32_t lo = odd ? got : ev, hi = odd ? od : got;  // key blocks 2m, 2m + 1
                kbits[m >> 3] |= (lo | (hi << 2)) << ((4 * m) & 31);
              }
            } else {
#pragma unroll 8
              for (int e = 0; e < 64; ++e) {
                const uint4 rr = philox4x32_10(make_uint4(kb0 + e, rb, uint32_t(h), uint32_t(b)),
                                               a.drop_k0, a.drop_k1);
                const uint32_t u0 = (grow & 1) ? rr.z : rr.x, u1 = (grow & 1) ? rr.w : rr.y;
                kbits[e >> 4] |= (uint32_t(u0 >= T) | (uint32_t(u1 >= T) << 1)) << ((2 * e) & 31);
              }
            }
          }
          uint32_t pk[2][32];
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            float2 t = ffma2(make_float2(x[2 * e], x[2 * e + 1]), cs, cm);
            t.x = ex2(t.x);
            t.y = ex2(t.y);
            s4[e & 3] = fadd2(s4[e & 3], t);
            if constexpr (DROP) {
              // the row sum above keeps the undropped values; 1/(1-p) goes in the epilogue
              const uint32_t kk = kbits[e >> 4] >> ((2 * e) & 31);
              pk[e >> 5][e & 31] = pack_bf16((kk & 1) ? t.x : 0.f, (kk & 2) ? t.y : 0.f);
            } else {
              pk[e >> 5][e & 31] = pack_bf16(t.x, t.y);
            }
          }
          const float2 s01 = fadd2(s4[0], s4[1]), s23 = fadd2(s4[2], s4[3]);
          const float2 st = fadd2(s01, s23);
          const float sum = st.x + st.y;
          l_run += sum;
          if (r == 0) BD_TRACE_EVENT(50 + s, int(tcount));  // softmax: exponentials done
          tmem_st32(tS, pk[0]);
          tmem_st32(tS + 32, pk[1]);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(B_PFULL + s));
          if (r == 0) BD_TRACE_EVENT(60 + s, int(tcount));  // softmax: P stored
          if (lane == 0) BD_TRACE_EVENT(4 * s + quarter, int(tcount));  // per warp: P stored
        }
        if (!ok) break;
        FwdUnit N;
        take(uk + 1, N);
        // the slot's warps meet at named barriers in the epilogue: leave together
        ok = bar_red_and(1 + s, 128, mbar_wait(bar(B_OFINAL + s), qi & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const float inv = (l_run > 0.f ? 1.f / l_run : 0.f) * (DROP ? a.drop_scale : 1.f);
        if constexpr (D <= 128) {
          // the whole O row leaves TMEM first, so that the next unit's first PV may
          // overwrite the accumulator while the row is stored
          uint32_t ov[D / 32][32];
#pragma unroll
          for (int q = 0; q < D / 32; ++q) tmem_ld32(tO + q * 32, ov[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < D / 32; ++q) reg_fence(ov[q]);
          tc_fence_before();
          mbar_arrive(bar(B_OEMPTY + s));
          // 64 columns at a time through the slot's staging box (row r's 16-byte
          // chunk c at c ^ (r & 7): the 128-byte swizzle of the map), sent by one
          // thread with a TMA store (rows past L are clipped); the threads' own row
          // stores kept the load/store unit busy through the next unit's start
          const uint32_t sbuf = sbase + Cfg::kOffStage + s * Cfg::kStageBytes;
#pragma unroll
          for (int k = 0; k < D / 64; ++k) {
            if (r == 0) bulk_wait_read<0>();  // the box sent from this buffer before has left it
            named_bar_sync(1 + s, 128);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              const uint32_t* v = ov[2 * k + (c8 >> 2)] + (c8 & 3) * 8;
              st_shared_v4(sbuf + r * 128 + ((c8 ^ (r & 7)) << 4),
                           pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                           pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                           pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                           pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + s, 128);
            if (r == 0) {
              tma_store_5d(&tm_o, sbuf, k * 64, h, U.qtile * 128, c, b);
              bulk_commit();
            }
          }
          if (row_ok) *lrow_p = l_run > 0.f ? (m_run + lg2(l_run)) * 0.69314718055994531f : -CUDART_INF_F;
        } else {
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(tO + q * 32, ov);
            tmem_ld_wait();
            reg_fence(ov);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
              for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
          }
          if (row_ok) *lrow_p = l_run > 0.f ? (m_run + lg2(l_run)) * 0.69314718055994531f : -CUDART_INF_F;
          tc_fence_before();
          mbar_arrive(bar(B_OEMPTY + s));
        }
        ++qi;
        U = N;
      }
      if (r == 0) bulk_wait<0>();  // the epilogue's TMA stores have completed
    }
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
      atomicExch(const_cast<int32_t*>(plan) + H_STATUS_DETAIL, 1);
    }
    unit_counters_release(claim, claim + 1);
  }
}

template <int D, bool DROP>
static int32_t launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                          const CUtensorMap& mo, const FwdArgs& a, int grid, cudaStream_t stream) {
  using Cfg = FwdCfg<D>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bd_fwd_kernel<D, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fwd)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, bd_fwd_kernel<D, DROP>);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(fwd)");
    // setmaxnreg.inc waits until registers are free: never launch a split that cannot be met
    if (fa.numRegs != Cfg::kRegsLaunch)
      return fail(BD_ERR_UNSUPPORTED, "fwd kernel built with %d registers/thread, its register split assumes %d",
                  fa.numRegs, Cfg::kRegsLaunch);
    attr_done[dev] = true;
  }
  bd_fwd_kernel<D, DROP><<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(mq, mk, mv, mo, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bd_fwd_kernel launch");
  return BD_OK;
}

}  // namespace bd

using namespace bd;

#ifdef BD_TRACE
// Trace build only: copies the [site][tile] clock table of CTA 0 to host memory
// (cap entries) and clears it; returns the number of entries copied.
extern "C" BD_API int32_t bd_trace_read(unsigned long long* host, int32_t cap) {
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

extern "C" int32_t bd_attn_fwd_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                                  const bd_tensor* k, const bd_tensor* v, int32_t row_offset, bd_tensor* out,
                                  bd_rowstat* lse, bd_tensor* dq_zero, void* stream) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!plan_dev || reinterpret_cast<uintptr_t>(plan_dev) % 16)
    return fail(BD_ERR_ARG, "plan_dev NULL or not 16-byte aligned");
  const int B = pv.hdr(H_B), C = pv.hdr(H_C), L = pv.hdr(H_L), H = pv.hdr(H_H), Hkv = pv.hdr(H_HKV);
  const int D = pv.hdr(H_D), Ck = pv.hdr(H_CK);
  if (row_offset >= 0) {
    if (pv.hdr(H_NITEMS) != B || C != 1)
      return fail(BD_ERR_PLAN, "row_offset given but the plan holds more than one chunk per sequence");
    for (int b = 0; b < B; ++b)
      if (pv.item(b)[I_ROW0] != row_offset)
        return fail(BD_ERR_PLAN, "row_offset %d differs from the plan's %d", row_offset, pv.item(b)[I_ROW0]);
  }
  if ((st = check_tensor(q, "q", 2, B, C, H, true))) return st;
  if ((st = check_tensor(k, "k", 2, B, Ck, Hkv, true))) return st;
  if ((st = check_tensor(v, "v", 2, B, Ck, Hkv, true))) return st;
  if ((st = check_tensor(out, "out", 2, B, C, H, false))) return st;
  if (!lse || !lse->ptr) return fail(BD_ERR_ARG, "lse: NULL");
  if (q->rows != L || out->rows != L) return fail(BD_ERR_ARG, "q/out rows must equal L = %d", L);
  if (k->rows < pv.hdr(H_KV_ROWS) || v->rows < pv.hdr(H_KV_ROWS))
    return fail(BD_ERR_ARG, "k/v rows %d/%d < %d needed by the plan", k->rows, v->rows, pv.hdr(H_KV_ROWS));
  if (reinterpret_cast<uintptr_t>(lse->ptr) % 4) return fail(BD_ERR_ALIGN, "lse not 4-byte aligned");
  if (dq_zero) {
    if ((st = check_tensor(dq_zero, "dq_zero", 4, B, C, H, false))) return st;
    if (dq_zero->rows != L) return fail(BD_ERR_ARG, "dq_zero rows must equal L = %d", L);
  }
  CUtensorMap mq, mk, mv, mo;
  std::memset(&mo, 0, sizeof(mo));
  if ((st = make_tmap_bf16(&mq, q, B, C, H, D, "q"))) return st;
  if ((st = make_tmap_bf16(&mk, k, B, Ck, Hkv, D, "k"))) return st;
  if ((st = make_tmap_bf16(&mv, v, B, Ck, Hkv, D, "v"))) return st;
  FwdArgs a;
  a.plan = static_cast<const int32_t*>(plan_dev);
  a.o = static_cast<__nv_bfloat16*>(out->ptr);
  a.o_sb = out->stride_b; a.o_sc = out->stride_c; a.o_sr = out->stride_row; a.o_sh = out->stride_head;
  a.lse = lse->ptr; a.l_sb = lse->stride_b; a.l_sc = lse->stride_c; a.l_sh = lse->stride_head;
  a.L = L; a.n_work = pv.hdr(H_NFWD); a.slots = pv.hdr(H_SLOTS); a.Ck = Ck;
  a.dqz = dq_zero ? static_cast<float*>(dq_zero->ptr) : nullptr;
  a.z_sb = dq_zero ? dq_zero->stride_b : 0; a.z_sc = dq_zero ? dq_zero->stride_c : 0;
  a.z_sr = dq_zero ? dq_zero->stride_row : 0; a.z_sh = dq_zero ? dq_zero->stride_head : 0;
  a.B = B; a.C = C; a.H = H;
  // O leaves by TMA at head dims 64 / 128 (the checks above give the 16-byte
  // aligned base and strides a tensor map needs)
  if (D <= 128 && (st = make_tmap_bf16(&mo, out, B, C, H, D, "o"))) return st;
  // each launch takes the next counter slot: launches sharing the device plan may
  // then overlap on the GPU (up to kFwdCounterSlots at once) without taking each
  // other's work units
  static std::atomic<uint32_t> launch_seq{0};
  a.counter_slot = int32_t(launch_seq.fetch_add(1, std::memory_order_relaxed) % kFwdCounterSlots);
  float scale;
  const int32_t scale_bits = pv.hdr(H_SCALE_BITS);
  memcpy(&scale, &scale_bits, 4);
  a.scale_log2 = scale * 1.4426950408889634f;
  if (a.n_work == 0) return ok();
  int nsm = 0;
  if ((st = sm_count(&nsm))) return st;
  const int grid = a.n_work < nsm ? a.n_work : nsm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  a.drop_thresh = uint32_t(pv.hdr(H_DROP_THRESH));
  a.drop_k0 = uint32_t(pv.hdr(H_DROP_SEED_LO));
  a.drop_k1 = uint32_t(pv.hdr(H_DROP_SEED_HI));
  const int32_t dbits = pv.hdr(H_DROP_SCALE_BITS);
  memcpy(&a.drop_scale, &dbits, 4);
  if (D == 256 && a.slots != 1) return fail(BD_ERR_PLAN, "head dim 256 plans use one query head per CTA");
  if (a.drop_thresh != 0)
    st = D == 256   ? launch_fwd<256, true>(mq, mk, mv, mo, a, grid, s)
         : D == 128 ? launch_fwd<128, true>(mq, mk, mv, mo, a, grid, s)
                    : launch_fwd<64, true>(mq, mk, mv, mo, a, grid, s);
  else
    st = D == 256   ? launch_fwd<256, false>(mq, mk, mv, mo, a, grid, s)
         : D == 128 ? launch_fwd<128, false>(mq, mk, mv, mo, a, grid, s)
                    : launch_fwd<64, false>(mq, mk, mv, mo, a, grid, s);
  if (st) return st;
  return ok();
}

extern "C" int32_t bd_attn_fwd(const void* plan_host, const void* plan_dev, const bd_tensor* q, const bd_tensor* k,
                               const bd_tensor* v, int32_t row_offset, bd_tensor* out, bd_rowstat* lse,
                               void* stream) {
  return bd_attn_fwd_ex(plan_host, plan_dev, q, k, v, row_offset, out, lse, nullptr, stream);
}
