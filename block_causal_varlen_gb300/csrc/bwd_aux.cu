// Small HBM-bound kernels around the backward main loop, plus status readback.
//
//   bd_bwd_pre_kernel   D_i = <dO_i, O_i> in fp32 for every (row, head) of every
//                       chunk and the log2-domain LSE; zeroes the main
//                       kernel's claim counters and (on request) the fp32 dQ
//                       accumulator rows.
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

using namespace dev;

BwdWorkspace bwd_workspace_layout(int nitems, int H, int Lpad) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdWorkspace w;
  const size_t stat = al(size_t(nitems) * H * Lpad * sizeof(float));
  w.lse2 = 0;
  w.dstat = stat;
  // the main kernel's work-unit claim counters live in the caller's workspace, so
  // backward launches that share a device plan but not a workspace may overlap
  w.counters = 2 * stat;
  w.total = w.counters + 256;
  return w;
}

namespace {

constexpr int kPreCtasPerSm = 3;                // CTAs resident per SM (their serial paths overlap)
constexpr int kPreStages = 4;                   // O + dO boxes in flight per CTA
constexpr int kPreBoxBytes = 8192;              // one O (or dO) box
constexpr int kPreStageBytes = 2 * kPreBoxBytes;
constexpr int kPreConsumers = 256;              // the dot-product warps; the next warp issues the loads
constexpr int kPreThreads = kPreConsumers + 32;
constexpr int kPrePieces = kPreBoxBytes / 16 / kPreConsumers;  // 16-byte pieces per consumer thread and box
constexpr int kPreAhead = 4;                    // LSE ring: loads issued kPreAhead - 1 groups ahead
constexpr int kPreOffBar = kPreStages * kPreStageBytes;
constexpr int kPreSmem = kPreOffBar + 2 * kPreStages * 8 + 16 + 1024;  // + alignment slack

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// Read-only global loads kept where they are written (volatile): issued ahead of
// the waits they are meant to overlap, not moved next to their first use.
__device__ __forceinline__ float ld_ahead_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int32_t ld_ahead_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Walks groups g, g + stride, g + 2 stride, ... as (item, row block, head block),
// group = (item * row_blocks + row block) * head_blocks + head block, by mixed-radix
// addition instead of a division per step.
struct PreIter {
  int hb, rb, item, dhb, drb, ditem, hbs, nrb;
  __device__ void init(const BwdPreArgs& a, int g, int stride) {
    hbs = a.head_blocks;
    nrb = a.Lpad / a.rows;
    hb = g % hbs;
    const int t = g / hbs;
    rb = t % nrb;
    item = t / nrb;
    dhb = stride % hbs;
    const int ts = stride / hbs;
    drb = ts % nrb;
    ditem = ts / nrb;
  }
  __device__ void next() {
    hb += dhb;
    int carry = 0;
    if (hb >= hbs) { hb -= hbs; carry = 1; }
    rb += drb + carry;
    carry = 0;
    if (rb >= nrb) { rb -= nrb; carry = 1; }
    item += ditem + carry;
  }
};

}  // namespace

// D_i = <dO_i, O_i> for every (row, head) of every chunk, the log2-domain LSE
// (+inf on rows without a document, where D is 0), the main kernel's claim
// counters zeroed and, unless the caller cleared it already, the fp32 dQ
// accumulator zeroed. A streaming kernel: kPreCtasPerSm CTAs per SM walk the
// groups blockIdx.x, blockIdx.x + gridDim.x, ...; a CTA's last warp brings each
// group's O and dO boxes into a ring of shared-memory stages by TMA (none for
// groups whose rows are all padding: live rows of an item are [0, L - npad)), and
// the warps below it take the dot products from shared memory, a (row, head)'s
// 16-byte pieces in
// D / 8 consecutive lanes summed with shuffles. The LSE values of a group are
// loaded kPreAhead - 1 groups ahead so that their latency stays off the stream.
template <int D>
__global__ void __launch_bounds__(kPreThreads, kPreCtasPerSm)
    bd_bwd_pre_kernel(const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_do,
                      BwdPreArgs a) {
  constexpr int CPH = D / 8;  // 16-byte pieces per head-row (8, 16 or 32: never straddle a warp)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  auto full = [&](int s) { return sbase + kPreOffBar + 8u * s; };
  auto empty = [&](int s) { return sbase + kPreOffBar + 8u * (kPreStages + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kPreOffBar + 16 * kPreStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* items = a.plan + a.items_off;
  const int grid = int(gridDim.x), bid = int(blockIdx.x);
  // this CTA's groups: bid + k * grid for k < niters
  const int niters = a.ngroups > bid ? (a.ngroups - bid + grid - 1) / grid : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPreStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kPreConsumers / 32);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (bid == 0 && threadIdx.x < 2) a.counters[threadIdx.x] = 0;
  __syncthreads();
  bool ok = true;

  if (warp == kPreConsumers / 32) {
    // ---- loads: lane j finds out whether group k + j has a live row, 32 groups at
    // a time (the next 32 groups' npad loaded while these are issued); lane 0 issues
    const uint32_t tx = uint32_t(2 * a.rows * a.heads * D * 2);
    if (lane == 0) {
      tma_prefetch_desc(&tm_o);
      tma_prefetch_desc(&tm_do);
    }
    PreIter li, it0;
    li.init(a, bid + lane * grid, 32 * grid);  // lane's group of the current batch
    it0.init(a, bid, grid);                    // lane 0's next group to issue
    int np = lane < niters ? ld_ahead_s32(items + li.item * kItemWords + I_NPAD) : 0;
    int issued = 0, s = 0;
    uint32_t phase = 0;
    for (int kb = 0; kb < niters && ok; kb += 32) {
      PreIter ln = li;
      ln.next();
      const int np_next = kb + 32 + lane < niters ? ld_ahead_s32(items + ln.item * kItemWords + I_NPAD) : 0;
      const bool live = kb + lane < niters && li.rb * a.rows < a.L - np;
      const uint32_t live_mask = __ballot_sync(0xffffffffu, live);
      if (lane == 0) {
        const int n = min(32, niters - kb);
        for (int j = 0; j < n; ++j) {
          const int k = kb + j;
          if (k >= kPreStages && !(ok = mbar_wait(empty(s), phase ^ 1u, abort_flag))) break;
          if ((live_mask >> j) & 1u) {
            const int b = it0.item / a.C, c = it0.item - b * a.C;
            const uint32_t st = sbase + uint32_t(s) * kPreStageBytes;
            mbar_expect_tx(full(s), tx);
            tma_load_5d(st, &tm_o, full(s), 0, it0.hb * a.heads, it0.rb * a.rows, c, b);
            tma_load_5d(st + kPreBoxBytes, &tm_do, full(s), 0, it0.hb * a.heads, it0.rb * a.rows, c, b);
          } else {
            mbar_arrive(full(s));  // nothing to load: the consumers write the padding values
          }
          issued = k + 1;
          it0.next();
          if (++s == kPreStages) { s = 0; phase ^= 1u; }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      np = np_next;
      li = ln;
    }
    if (lane == 0 && !ok) {
      // stop only after the boxes already on their way have landed
      for (int k = max(0, issued - kPreStages); k < issued; ++k) mbar_wait_drain(full(k % kPreStages), (k / kPreStages) & 1);
    }
  } else {
    // ---- dot products: thread t takes pieces t + i * kPreConsumers of each
    // group's box, whose (row, head) within the box is the same for every group
    const int t = threadIdx.x;
    const int P = a.rows * a.heads * CPH;  // 16-byte pieces per box (<= 512)
    const float inf = __int_as_float(0x7f800000);
    int pr[kPrePieces], ph[kPrePieces];
    bool lead[kPrePieces];
#pragma unroll
    for (int i = 0; i < kPrePieces; ++i) {
      const int p = t + i * kPreConsumers, rh = p / CPH;
      lead[i] = p < P && p % CPH == 0;
      pr[i] = rh / a.heads;
      ph[i] = rh % a.heads;
    }
    float lring[kPreAhead][kPrePieces];
    int nring[kPreAhead];
    PreIter cur, ahead;
    cur.init(a, bid, grid);
    ahead = cur;
    auto prefetch = [&](int k, float (&lv)[kPrePieces], int& npad) {
#pragma unroll
      for (int i = 0; i < kPrePieces; ++i) lv[i] = 0.f;
      npad = 0;
      if (k < niters) {
        npad = ld_ahead_s32(items + ahead.item * kItemWords + I_NPAD);
        const int b = ahead.item / a.C, c = ahead.item - b * a.C;
        const float* base = a.lse + b * a.l_sb + c * a.l_sc;
#pragma unroll
        for (int i = 0; i < kPrePieces; ++i) {
          const int h = ahead.hb * a.heads + ph[i], l = ahead.rb * a.rows + pr[i];
          if (lead[i] && h < a.H && l < a.L) lv[i] = ld_ahead_f32(base + int64_t(h) * a.l_sh + l);
        }
      }
      ahead.next();
    };
#pragma unroll
    for (int j = 0; j < kPreAhead - 1; ++j) prefetch(j, lring[j], nring[j]);
    int s = 0;
    uint32_t phase = 0;
    for (int k0 = 0; k0 < niters && ok; k0 += kPreAhead) {
#pragma unroll
      for (int j = 0; j < kPreAhead; ++j) {
        const int k = k0 + j;
        if (k >= niters) break;  // the same for every thread of the CTA
        prefetch(k + kPreAhead - 1, lring[(j + kPreAhead - 1) % kPreAhead], nring[(j + kPreAhead - 1) % kPreAhead]);
        const int l0 = cur.rb * a.rows, h0 = cur.hb * a.heads, item = cur.item;
        const int n_live = a.L - nring[j];
        const bool live = l0 < n_live;  // the same test the load warp made
        if (!(ok = mbar_wait(full(s), phase, abort_flag))) break;
        float acc[kPrePieces];
#pragma unroll
        for (int i = 0; i < kPrePieces; ++i) acc[i] = 0.f;
        if (live) {
          const uint32_t st = sbase + uint32_t(s) * kPreStageBytes;
#pragma unroll
          for (int i = 0; i < kPrePieces; ++i) {
            const int p = t + i * kPreConsumers;
            if (p < P) {
              const uint4 ov = ld_shared_u4(st + 16u * p), gv = ld_shared_u4(st + kPreBoxBytes + 16u * p);
              const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
              const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 x = __bfloat1622float2(o2[e]), y = __bfloat1622float2(g2[e]);
                acc[i] = fmaf(x.x, y.x, fmaf(x.y, y.y, acc[i]));
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == kPreStages) { s = 0; phase ^= 1u; }
#pragma unroll
        for (int i = 0; i < kPrePieces; ++i)
#pragma unroll
          for (int off = CPH / 2; off > 0; off >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
#pragma unroll
        for (int i = 0; i < kPrePieces; ++i) {
          const int h = h0 + ph[i], l = l0 + pr[i];
          if (lead[i] && h < a.H) {
            const bool rl = l < n_live;  // padding rows and rows past L: no attention
            const int64_t sidx = (int64_t(item) * a.H + h) * a.Lpad + l;
            a.dstat[sidx] = rl ? acc[i] : 0.f;
            a.lse2[sidx] = rl ? lring[j][i] * 1.4426950408889634f : inf;
          }
        }
        if (a.clear_dq) {
          const int b = item / a.C, c = item - b * a.C;
          for (int f = t; f < 2 * P; f += kPreConsumers) {
            const int rh = f / (D / 4), l = l0 + rh / a.heads, h = h0 + rh % a.heads, col = (f % (D / 4)) * 4;
            if (h < a.H && l < a.L)
              *reinterpret_cast<float4*>(a.dq + b * a.q_sb + c * a.q_sc + int64_t(l) * a.q_sr +
                                         int64_t(h) * a.q_sh + col) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        cur.next();
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    atomicExch(const_cast<int32_t*>(a.plan) + H_STATUS, DEV_TIMEOUT);
    atomicExch(const_cast<int32_t*>(a.plan) + H_STATUS_DETAIL, 4);
  }
}

int32_t launch_bwd_pre(const CUtensorMap& mo, const CUtensorMap& mdo, const BwdPreArgs& a, int D, cudaStream_t s) {
  if (a.ngroups == 0) return BD_OK;
  int nsm = 0;
  int32_t st = sm_count(&nsm);
  if (st) return st;
  const int grid = a.ngroups < kPreCtasPerSm * nsm ? a.ngroups : kPreCtasPerSm * nsm;
  static bool attr_done[64][3] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int di = D == 256 ? 2 : D == 128 ? 1 : 0;
  if (dev < 64 && !attr_done[dev][di]) {
    cudaError_t e = D == 256   ? cudaFuncSetAttribute(bd_bwd_pre_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreSmem)
                    : D == 128 ? cudaFuncSetAttribute(bd_bwd_pre_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreSmem)
                               : cudaFuncSetAttribute(bd_bwd_pre_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd pre)");
    attr_done[dev][di] = true;
  }
  if (D == 256) bd_bwd_pre_kernel<256><<<grid, kPreThreads, kPreSmem, s>>>(mo, mdo, a);
  else if (D == 128) bd_bwd_pre_kernel<128><<<grid, kPreThreads, kPreSmem, s>>>(mo, mdo, a);
  else bd_bwd_pre_kernel<64><<<grid, kPreThreads, kPreSmem, s>>>(mo, mdo, a);
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
