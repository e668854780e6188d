// Backward of block-causal varlen chunked attention on sm_103a (main loop: in progress).
#include <cuda_runtime.h>

#include "bwd_aux.h"
#include "host_util.h"
#include "plan_layout.h"

using namespace bd;

extern "C" int32_t bd_attn_bwd_workspace(const void* plan_host, size_t* bytes) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!bytes) return fail(BD_ERR_ARG, "bytes is NULL");
  const size_t n = size_t(pv.hdr(H_NITEMS)) * pv.hdr(H_H) * pv.hdr(H_L) * sizeof(float);
  *bytes = (n + 255) & ~size_t(255);
  return ok();
}

extern "C" int32_t bd_attn_bwd(const void* plan_host, const void* plan_dev, const bd_tensor* q, const bd_tensor* k,
                               const bd_tensor* v, const bd_tensor* out, const bd_tensor* dout,
                               const bd_rowstat* lse, bd_tensor* dq, bd_tensor* dk, bd_tensor* dv,
                               int32_t accumulate_dkv, void* workspace, size_t workspace_bytes, void* stream) {
  (void)plan_dev; (void)q; (void)k; (void)v; (void)out; (void)dout; (void)lse; (void)dq; (void)dk; (void)dv;
  (void)accumulate_dkv; (void)workspace; (void)workspace_bytes; (void)stream;
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  return fail(BD_ERR_UNSUPPORTED, "backward not built yet");
}
