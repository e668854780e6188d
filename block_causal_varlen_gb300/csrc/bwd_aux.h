// Argument blocks of the backward's auxiliary kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bd {

struct BwdPreArgs {
  const int32_t* plan;
  const float* lse;
  int64_t l_sb, l_sc, l_sh;
  float* lse2;     // workspace [nitems, H, Lpad]: LSE * log2(e), +inf on invalid rows
  float* dstat;    // workspace [nitems, H, Lpad]: D = <dO, O>
  int32_t* counters;  // workspace: the main kernel's (claim, done) work-unit counters, zeroed here
  float* dq;       // zeroed when clear_dq is set
  int64_t q_sb, q_sc, q_sr, q_sh;
  int32_t nitems, C, L, Lpad, H, clear_dq;
  int32_t items_off;  // word offset of the plan's chunk items
  // a group is `rows` consecutive rows x `heads` heads of one item: the O / dO box
  // one stage of the statistics kernel holds; groups are numbered
  // ((item * (Lpad / rows) + row block) * head_blocks + head block)
  int32_t rows, heads, head_blocks, ngroups;
};

// Workspace layout of the backward (offsets in bytes, 256-byte aligned).
struct BwdWorkspace {
  size_t lse2, dstat, counters, total;
};
BwdWorkspace bwd_workspace_layout(int nitems, int H, int Lpad);

struct OwnerSumArgs {
  const int32_t* plan;
  const float* dk_win;
  const float* dv_win;
  float* dk;
  float* dv;
  int64_t wk_sb, wk_sc, wk_sr, wk_sh, wv_sb, wv_sc, wv_sr, wv_sh;
  int64_t k_sb, k_sr, k_sh, v_sb, v_sr, v_sh;
  int32_t B, C, S, Hkv, d;
  int32_t accumulate;  // 1: add the sum into dk / dv; 0: overwrite them with it
};

// Launches the statistics kernel over maps of O and dO with the args' row box.
int32_t launch_bwd_pre(const CUtensorMap& mo, const CUtensorMap& mdo, const BwdPreArgs& a, int D, cudaStream_t s);

}  // namespace bd
