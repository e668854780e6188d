// Small HBM-bound kernels around the backward main loop, plus status readback.
//
//   bd_bwd_pre_kernel   D_i = <dO_i, O_i> in fp32 for every (row, head) of every
//                       chunk, the log2-domain LSE and each row's document
//                       start, and zeroes the fp32 dQ accumulator rows.
//   bd_owner_sum_kernel adds needed-only-window dK/dV partials into the rows'
//                       owners, chunk by chunk in plan order (deterministic);
//                       the single-GPU form of the index_add / reduce-scatter
//                       SUM backward of the needed-only exchange (NeMo
//                       Automodel page "block-diagonal varlen CP for packed
//                       sequences", Design overview, exchange.py).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd_aux.h"
#include "host_util.h"
#include "plan_layout.h"
#include "ptx.cuh"

namespace bd {

BwdWorkspace bwd_workspace_layout(int nitems, int H, int Lpad) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdWorkspace w;
  const size_t stat = al(size_t(nitems) * H * Lpad * sizeof(float));
  w.lse2 = 0;
  w.dstat = stat;
  w.rowds = 2 * stat;
  // the main kernel's work-unit claim counters live in the caller's workspace, so
  // backward launches that share a device plan but not a workspace may overlap
  w.counters = 2 * stat + al(size_t(nitems) * Lpad * sizeof(int32_t));
  w.total = w.counters + 256;
  return w;
}

// One block per `rows_per_block` consecutive rows (1, 2 or 4; they divide Lpad, so
// a block's rows belong to one item): D for every head, the log2-domain LSE, the
// row's document start, and (unless the caller cleared it already) zeroing of the
// row's dQ accumulator. Threads take 16-byte pieces of O / dO of all heads of
// the block's rows, up to four pieces each at a time, so that a thread keeps up
// to 64 bytes of loads in flight; a head's pieces sit in consecutive lanes and
// are summed with shuffles. Padding rows (no document) read nothing: their D is
// 0 and their log2 LSE +inf.
template <int D>
__global__ void __launch_bounds__(256) bd_bwd_pre_kernel(BwdPreArgs a) {
  constexpr int CPH = D / 8;  // 16-byte pieces per head (8, 16 or 32: groups never straddle a warp)
  const int R = a.rows_per_block;
  const int64_t grow0 = int64_t(blockIdx.x) * R;  // first row of the block in [nitems, Lpad]
  const int item = int(grow0 / a.Lpad), l0 = int(grow0 % a.Lpad);
  const int b = item / a.C, c = item % a.C;
  const int tid = threadIdx.x;
  if (blockIdx.x == 0 && tid < 2) a.counters[tid] = 0;  // the main kernel's claim counters
  const float inf = __int_as_float(0x7f800000);
  __shared__ int s_ds[4];
  if (tid < R) {
    const int l = l0 + tid;
    int32_t v = 0x7fffffff;
    if (l < a.L) v = a.plan[a.rowds_off + int64_t(item) * a.Lpad + l];
    a.rowds[int64_t(item) * a.Lpad + l] = v;
    s_ds[tid] = v == kRowInvalid ? -1 : v;
  }
  if (a.clear_dq) {
    const int per_row = a.H * (D / 4);
    for (int f = tid; f < R * per_row; f += 256) {
      const int r = f / per_row, k = f % per_row;
      const int l = l0 + r;
      if (l >= a.L) continue;
      const int h = k / (D / 4), col = (k % (D / 4)) * 4;
      float* p = a.dq + b * a.q_sb + c * a.q_sc + int64_t(l) * a.q_sr + int64_t(h) * a.q_sh + col;
      *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  const int npieces = a.H * CPH;  // per row
  const int total = R * npieces;
  for (int f0 = 0; f0 < total; f0 += 1024) {
    uint4 ov[4], gv[4];
    float lv[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int f = f0 + rr * 256 + tid;
      ov[rr] = gv[rr] = make_uint4(0u, 0u, 0u, 0u);
      lv[rr] = 0.f;
      if (f < total) {
        const int r = f / npieces, k = f % npieces;
        if (s_ds[r] >= 0) {
          const int l = l0 + r, h = k / CPH, col = (k % CPH) * 8;
          ov[rr] = *reinterpret_cast<const uint4*>(a.o + b * a.o_sb + c * a.o_sc + int64_t(l) * a.o_sr +
                                                   int64_t(h) * a.o_sh + col);
          gv[rr] = *reinterpret_cast<const uint4*>(a.dout + b * a.g_sb + c * a.g_sc + int64_t(l) * a.g_sr +
                                                   int64_t(h) * a.g_sh + col);
          if (k % CPH == 0) lv[rr] = a.lse[b * a.l_sb + c * a.l_sc + int64_t(h) * a.l_sh + l];
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      if (f0 + rr * 256 >= total) break;  // the same for the whole block: every lane shuffles
      const int f = f0 + rr * 256 + tid;
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[rr]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[rr]);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(o2[i]), y = __bfloat1622float2(g2[i]);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
      }
#pragma unroll
      for (int off = CPH / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (f < total && (f % CPH) == 0) {
        const int r = f / npieces, h = (f % npieces) / CPH;
        const bool live = s_ds[r] >= 0;  // padding rows and rows past L: no attention
        const int64_t sidx = (int64_t(item) * a.H + h) * a.Lpad + l0 + r;
        a.dstat[sidx] = live ? acc : 0.f;
        a.lse2[sidx] = live ? lv[rr] * 1.4426950408889634f : inf;
      }
    }
  }
}

int32_t launch_bwd_pre(const BwdPreArgs& a, int D, cudaStream_t s) {
  const int64_t blocks = int64_t(a.nitems) * a.Lpad / a.rows_per_block;
  if (blocks == 0) return BD_OK;
  if (blocks > 0x7fffffff) return fail(BD_ERR_UNSUPPORTED, "too many rows for the statistics kernel");
  if (D == 256) bd_bwd_pre_kernel<256><<<unsigned(blocks), 256, 0, s>>>(a);
  else if (D == 128) bd_bwd_pre_kernel<128><<<unsigned(blocks), 256, 0, s>>>(a);
  else bd_bwd_pre_kernel<64><<<unsigned(blocks), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? BD_OK : cuda_fail(e, "bd_bwd_pre_kernel launch");
}

// One thread per (b, global row, head, 4 columns): sums the chunks' windows in order
// and adds the sum into the owner row, or stores it there (every owner row is
// written, rows no window covers with zeros).
__global__ void __launch_bounds__(256) bd_owner_sum_kernel(OwnerSumArgs a) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int q4 = a.d / 4;
  const int64_t total = int64_t(a.B) * a.S * a.Hkv * q4;
  if (t >= total) return;
  const int col = int(t % q4) * 4;
  const int h = int((t / q4) % a.Hkv);
  const int row = int((t / (int64_t(q4) * a.Hkv)) % a.S);
  const int b = int(t / (int64_t(q4) * a.Hkv * a.S));
  const int32_t* items = a.plan + a.plan[H_OFF_ITEMS];
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
  for (int c = 0; c < a.C; ++c) {
    const int32_t* I = items + (b * a.C + c) * kItemWords;
    const int r = row - I[I_KVSTART];
    if (row < I[I_KVSTART] || row >= I[I_KVEND]) continue;
    const int64_t off_k = b * a.wk_sb + c * a.wk_sc + int64_t(r) * a.wk_sr + int64_t(h) * a.wk_sh + col;
    const int64_t off_v = b * a.wv_sb + c * a.wv_sc + int64_t(r) * a.wv_sr + int64_t(h) * a.wv_sh + col;
    const float4 x = *reinterpret_cast<const float4*>(a.dk_win + off_k);
    const float4 y = *reinterpret_cast<const float4*>(a.dv_win + off_v);
    sk.x += x.x; sk.y += x.y; sk.z += x.z; sk.w += x.w;
    sv.x += y.x; sv.y += y.y; sv.z += y.z; sv.w += y.w;
  }
  float4* pk = reinterpret_cast<float4*>(a.dk + b * a.k_sb + int64_t(row) * a.k_sr + int64_t(h) * a.k_sh + col);
  float4* pv = reinterpret_cast<float4*>(a.dv + b * a.v_sb + int64_t(row) * a.v_sr + int64_t(h) * a.v_sh + col);
  if (a.accumulate) {
    const float4 ok = *pk, ov = *pv;
    sk.x += ok.x; sk.y += ok.y; sk.z += ok.z; sk.w += ok.w;
    sv.x += ov.x; sv.y += ov.y; sv.z += ov.z; sv.w += ov.w;
  }
  *pk = sk;
  *pv = sv;
}

// Waits, with the kernels' bounded wait, on an mbarrier that nothing arrives at,
// then records the timeout in the plan's status word like any kernel would.
__global__ void bd_selftest_wait_kernel(int32_t* plan, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t mbar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    dev::mbar_init(dev::smem_u32(&mbar), 1);
    abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  const bool ok = dev::mbar_wait(dev::smem_u32(&mbar), 0, &abort_flag, limit_ns);
  if (!ok && threadIdx.x == 0) {
    atomicExch(plan + H_STATUS, DEV_TIMEOUT);
    atomicExch(plan + H_STATUS_DETAIL, 99);
  }
}

}  // namespace bd

using namespace bd;

extern "C" int32_t bd_selftest_bounded_wait(const void* plan_dev, uint32_t limit_us, void* stream) {
  if (!plan_dev || reinterpret_cast<uintptr_t>(plan_dev) % 16) return fail(BD_ERR_ARG, "plan_dev NULL/misaligned");
  if (limit_us == 0 || limit_us > 1000000) return fail(BD_ERR_ARG, "limit_us must be in (0, 1e6]");
  bd_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      const_cast<int32_t*>(static_cast<const int32_t*>(plan_dev)), uint64_t(limit_us) * 1000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bd_selftest_wait_kernel launch");
  return ok();
}

extern "C" int32_t bd_owner_sum_ex(const void* plan_host, const void* plan_dev, const bd_tensor* dk_win,
                                   const bd_tensor* dv_win, bd_tensor* dk, bd_tensor* dv, int32_t accumulate,
                                   void* stream) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!plan_dev) return fail(BD_ERR_ARG, "plan_dev is NULL");
  if (pv.hdr(H_KVMODE) != BD_KV_WINDOW) return fail(BD_ERR_PLAN, "bd_owner_sum needs a BD_KV_WINDOW plan");
  const int B = pv.hdr(H_B), C = pv.hdr(H_C), Hkv = pv.hdr(H_HKV), S = pv.hdr(H_S), D = pv.hdr(H_D);
  if ((st = check_tensor(dk_win, "dk_win", 4, B, C, Hkv, false))) return st;
  if ((st = check_tensor(dv_win, "dv_win", 4, B, C, Hkv, false))) return st;
  if ((st = check_tensor(dk, "dk", 4, B, 1, Hkv, false))) return st;
  if ((st = check_tensor(dv, "dv", 4, B, 1, Hkv, false))) return st;
  if (dk->rows < S || dv->rows < S) return fail(BD_ERR_ARG, "dk/dv rows must be >= S = %d", S);
  if (dk_win->rows < pv.hdr(H_KV_ROWS) || dv_win->rows < pv.hdr(H_KV_ROWS))
    return fail(BD_ERR_ARG, "window rows < %d", pv.hdr(H_KV_ROWS));
  OwnerSumArgs a;
  a.plan = static_cast<const int32_t*>(plan_dev);
  a.dk_win = static_cast<const float*>(dk_win->ptr);
  a.dv_win = static_cast<const float*>(dv_win->ptr);
  a.dk = static_cast<float*>(dk->ptr);
  a.dv = static_cast<float*>(dv->ptr);
  a.wk_sb = dk_win->stride_b; a.wk_sc = dk_win->stride_c; a.wk_sr = dk_win->stride_row; a.wk_sh = dk_win->stride_head;
  a.wv_sb = dv_win->stride_b; a.wv_sc = dv_win->stride_c; a.wv_sr = dv_win->stride_row; a.wv_sh = dv_win->stride_head;
  a.k_sb = dk->stride_b; a.k_sr = dk->stride_row; a.k_sh = dk->stride_head;
  a.v_sb = dv->stride_b; a.v_sr = dv->stride_row; a.v_sh = dv->stride_head;
  a.B = B; a.C = C; a.S = S; a.Hkv = Hkv; a.d = D; a.accumulate = accumulate ? 1 : 0;
  const int64_t total = int64_t(B) * S * Hkv * (D / 4);
  bd_owner_sum_kernel<<<unsigned((total + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bd_owner_sum_kernel launch");
  return ok();
}

extern "C" int32_t bd_owner_sum(const void* plan_host, const void* plan_dev, const bd_tensor* dk_win,
                                const bd_tensor* dv_win, bd_tensor* dk, bd_tensor* dv, void* stream) {
  return bd_owner_sum_ex(plan_host, plan_dev, dk_win, dv_win, dk, dv, 1, stream);
}

extern "C" int32_t bd_check_status(const void* plan_dev, int32_t reset, void* stream) {
  if (!plan_dev) return fail(BD_ERR_ARG, "plan_dev is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host[2] = {0, 0};
  const int32_t* p = static_cast<const int32_t*>(plan_dev) + H_STATUS;
  cudaError_t e = cudaMemcpyAsync(host, p, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "bd_check_status readback");
  if (reset && (host[0] || host[1])) {
    e = cudaMemsetAsync(const_cast<int32_t*>(p), 0, sizeof(host), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "bd_check_status reset");
  }
  if (host[0] == DEV_TIMEOUT)
    return fail(BD_ERR_DEVICE_TIMEOUT, "a kernel stopped after a bounded wait timed out (site %d)", host[1]);
  if (host[0] == DEV_SMEM_ALIGN)
    return fail(BD_ERR_CUDA, "a kernel found its shared memory not 1024-byte aligned and did no work (site %d)",
                host[1]);
  if (host[0] != DEV_OK) return fail(BD_ERR_CUDA, "a kernel recorded failure code %d (site %d)", host[0], host[1]);
  return ok();
}
