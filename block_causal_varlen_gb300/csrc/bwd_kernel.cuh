// Pieces shared by the backward main kernels (head dim 64 / 128 in attn_bwd.cu,
// head dim 256 in attn_bwd256.cu): their argument block, the order in which
// every role walks a work unit's steps, and the head dim 256 launcher.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan_layout.h"

namespace bd {

struct BwdArgs {
  const int32_t* plan;
  const float* lse2;
  const float* dstat;
  const int32_t* rowds;  // the plan's per-row document starts, [nitems][Lpad]
  int32_t* counters;  // (claim, done) work-unit counters in the workspace
  float* dq;
  int64_t q_sb, q_sc, q_sr, q_sh;
  float* dk;
  int64_t k_sb, k_sc, k_sr, k_sh;
  float* dv;
  int64_t v_sb, v_sc, v_sr, v_sh;
  int32_t L, Lpad, H, G, Ck, n_work, accumulate, dk_rows;
  int32_t work_off;  // plan word offset of the work-unit list the launch walks
  int32_t ck_out;    // chunk extent of the dK / dV output (its buffer index = b * ck_out + c)
  float scale, scale_log2;
  // attention dropout (used by the DROP instantiations): keep iff Philox word >= thresh
  uint32_t drop_thresh, drop_k0, drop_k1;
  float drop_scale;
};

// Iterates the (item, query step, head) steps of a backward work unit in the
// same order for every role; a query step is QR rows of one chunk.
template <int QR>
struct StepRange {
  const int32_t* items;
  int it_lo, it_hi, q_lo, q_hi, L;
  __device__ bool tiles(int it, int& t0, int& t1, int& r0) const {
    const int32_t* I = items + it * kItemWords;
    r0 = I[I_ROW0];
    const int lo = max(q_lo, r0), hi = min(q_hi, r0 + L);
    if (lo >= hi) return false;
    t0 = (lo - r0) / QR;
    t1 = (hi - 1 - r0) / QR;
    return true;
  }
};

// Launches the head dim 256 backward main kernel (maps: Q and dO with 64-row
// boxes, K and V with 128-row boxes, dQ with 16-row x 32-column reduce boxes).
int32_t launch_bwd256(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                      const CUtensorMap& mdq, const BwdArgs& a, bool drop, int grid, cudaStream_t stream);

}  // namespace bd
