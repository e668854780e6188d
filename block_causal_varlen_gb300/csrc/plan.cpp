// Host side of libbd: varlen segmentation of a context-parallel chunk, the
// plan blob the kernels consume, and error reporting.
//
// Segmentation follows the NeMo Automodel page "block-diagonal varlen CP for
// packed sequences": batch.py pads S to a multiple of cp and gives rank r the
// contiguous rows [r*L, (r+1)*L) and precomputes the varlen metadata once per
// step (Design overview; Summary, "zero per-layer host syncs"); kernels.py
// cuts the chunk into one segment per overlapping document and validates every
// offset on the host (Design overview; Key correctness property 4); a document
// straddling the chunk's left edge yields a segment with K longer than Q and
// bottom-right causal alignment (Key correctness property 2); the needed-only
// K/V window starts at the first document the chunk overlaps (Summary).
// Segments come from cu_seqlens by binary search.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.h"
#include "plan_layout.h"

namespace bd {

static thread_local std::string g_last_error;

int32_t fail(int32_t status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int32_t ok() {
  g_last_error.clear();
  return BD_OK;
}

const int32_t* PlanView::item(int i) const { return w + w[H_OFF_ITEMS] + i * kItemWords; }
const int32_t* PlanView::seg(int i) const { return w + w[H_OFF_SEGS] + i * kSegWords; }
const int32_t* PlanView::fwd(int i) const { return w + w[H_OFF_FWD] + i * kFwdWords; }
const int32_t* PlanView::bwd(int i) const { return w + w[H_OFF_BWD] + i * kBwdWords; }

int32_t view_plan(const void* plan_host, PlanView* out) {
  if (!plan_host) return fail(BD_ERR_ARG, "plan_host is NULL");
  const int32_t* w = static_cast<const int32_t*>(plan_host);
  if (w[H_MAGIC] != kPlanMagic || w[H_VERSION] != kPlanVersion)
    return fail(BD_ERR_PLAN, "plan blob has a bad magic/version");
  const int64_t words = w[H_WORDS];
  auto in = [&](int64_t off, int64_t n, int stride) {
    return off >= kHdrWords && n >= 0 && off + n * stride <= words;
  };
  if (!in(w[H_OFF_ITEMS], w[H_NITEMS], kItemWords) || !in(w[H_OFF_SEGS], w[H_NSEGS], kSegWords) ||
      !in(w[H_OFF_FWD], w[H_NFWD], kFwdWords) || !in(w[H_OFF_BWD], w[H_NBWD], kBwdWords) ||
      (w[H_NBWDO] != 0 && !in(w[H_OFF_BWDO], w[H_NBWDO], kBwdWords)) ||
      !in(w[H_OFF_ROWDS], w[H_NITEMS], int64_t(w[H_QTILES]) * kTile))
    return fail(BD_ERR_PLAN, "plan blob offsets are inconsistent");
  out->w = w;
  return BD_OK;
}

}  // namespace bd

using namespace bd;

extern "C" const char* bd_last_error(void) { return g_last_error.c_str(); }

extern "C" int32_t bd_version(void) { return 100; }

extern "C" int32_t bd_padded_len(int32_t s, int32_t cp) {
  if (s < 0 || cp <= 0) return fail(BD_ERR_ARG, "bd_padded_len: s < 0 or cp <= 0");
  return ((s + cp - 1) / cp) * cp;
}

static int32_t validate_cu(const int32_t* cu, int32_t ndocs, int32_t S) {
  if (!cu) return fail(BD_ERR_ARG, "cu_seqlens is NULL");
  if (ndocs < 0) return fail(BD_ERR_ARG, "ndocs < 0");
  if (S <= 0) return fail(BD_ERR_ARG, "S must be positive");
  if (cu[0] != 0) return fail(BD_ERR_CU_SEQLENS, "cu_seqlens[0] = %d, expected 0", cu[0]);
  for (int32_t i = 0; i < ndocs; ++i)
    if (cu[i + 1] < cu[i])
      return fail(BD_ERR_CU_SEQLENS, "cu_seqlens decreases at %d (%d -> %d)", i, cu[i], cu[i + 1]);
  if (cu[ndocs] > S)
    return fail(BD_ERR_CU_SEQLENS, "cu_seqlens[%d] = %d exceeds S = %d", ndocs, cu[ndocs], S);
  return BD_OK;
}

extern "C" int32_t bd_segment(const int32_t* cu, int32_t ndocs, int32_t S, int32_t cp, int32_t rank,
                              bd_chunk_hdr* hdr, bd_segment_t* segs, int32_t seg_capacity) {
  if (!hdr) return fail(BD_ERR_ARG, "hdr is NULL");
  int32_t st = validate_cu(cu, ndocs, S);
  if (st) return st;
  if (cp <= 0) return fail(BD_ERR_ARG, "cp must be positive");
  if (S % cp != 0) return fail(BD_ERR_NOT_DIVISIBLE, "S = %d is not a multiple of cp = %d", S, cp);
  if (rank < 0 || rank >= cp) return fail(BD_ERR_RANK, "rank %d outside [0, %d)", rank, cp);
  if (segs && seg_capacity < 0) return fail(BD_ERR_ARG, "seg_capacity < 0");

  const int32_t L = S / cp, row0 = rank * L, s_valid = cu[ndocs];
  const int32_t q_lo = row0, q_hi = std::min(row0 + L, s_valid);
  bd_chunk_hdr h;
  h.S = S; h.cp = cp; h.rank = rank; h.L = L; h.row_offset = row0; h.s_valid = s_valid;
  h.nseg = 0;
  h.n_pad = L - std::max(0, q_hi - q_lo);
  h.kv_start = h.kv_end = std::min(row0, s_valid);
  int32_t n = 0;
  if (q_lo < q_hi) {
    // first document whose end lies past q_lo
    const int32_t* first = std::upper_bound(cu + 1, cu + ndocs + 1, q_lo);
    for (int32_t doc = int32_t(first - (cu + 1)); doc < ndocs && cu[doc] < q_hi; ++doc) {
      const int32_t qs = std::max(cu[doc], q_lo), qe = std::min(cu[doc + 1], q_hi);
      if (qe <= qs) continue;  // zero-length document
      if (n == 0) h.kv_start = cu[doc];
      if (segs && n < seg_capacity) {
        bd_segment_t& s = segs[n];
        s.doc = doc; s.q_start = qs; s.q_len = qe - qs; s.k_start = cu[doc];
        s.k_len = qe - cu[doc]; s.diag_off = s.k_len - s.q_len;
      }
      ++n;
    }
    h.kv_end = q_hi;
  }
  h.nseg = n;
  *hdr = h;
  if (segs && n > seg_capacity)
    return fail(BD_ERR_CAPACITY, "chunk has %d segments, capacity %d", n, seg_capacity);
  return ok();
}

extern "C" int32_t bd_doc_ids_to_cu(const int32_t* ids, int32_t n, int32_t* cu_out, int32_t cap,
                                    int32_t* ndocs_out) {
  if (!ids || !ndocs_out || n < 0) return fail(BD_ERR_ARG, "doc_ids / ndocs_out NULL or n < 0");
  int32_t valid = 0;
  while (valid < n && ids[valid] >= 0) ++valid;
  for (int32_t t = valid; t < n; ++t)
    if (ids[t] >= 0) return fail(BD_ERR_CU_SEQLENS, "padding (negative id) at %d is not a suffix", valid);
  int32_t nd = 0;
  for (int32_t t = 0; t < valid; ++t) {
    if (t > 0 && ids[t] < ids[t - 1])
      return fail(BD_ERR_CU_SEQLENS, "document ids decrease at token %d (%d -> %d)", t, ids[t - 1], ids[t]);
    if (t == 0 || ids[t] != ids[t - 1]) ++nd;
  }
  *ndocs_out = nd;
  if (!cu_out || cap < nd + 1) return fail(BD_ERR_CAPACITY, "cu_out needs %d entries", nd + 1);
  int32_t k = 0;
  cu_out[k++] = 0;
  for (int32_t t = 1; t <= valid; ++t)
    if (t == valid || ids[t] != ids[t - 1]) cu_out[k++] = t;
  if (valid == 0) k = 1;
  return ok();
}

extern "C" int32_t bd_exchange_plan(const int32_t* cu, int32_t ndocs, int32_t S, int32_t cp, int32_t rank,
                                    int32_t* kind_out, bd_xfer_t* xfers, int32_t cap, int32_t* nxfer_out) {
  if (!kind_out || !nxfer_out) return fail(BD_ERR_ARG, "kind_out / nxfer_out NULL");
  bd_chunk_hdr h;
  int32_t st = bd_segment(cu, ndocs, S, cp, rank, &h, nullptr, 0);
  if (st) return st;
  const int32_t L = h.L;
  int32_t n = 0, remote_owners = 0;
  if (h.kv_end > h.kv_start) {
    for (int32_t o = h.kv_start / L; o <= (h.kv_end - 1) / L; ++o) {
      const int32_t lo = std::max(h.kv_start, o * L), hi = std::min(h.kv_end, (o + 1) * L);
      if (hi <= lo) continue;
      if (xfers && n < cap) {
        xfers[n].src_rank = o; xfers[n].src_row = lo; xfers[n].n_rows = hi - lo;
        xfers[n].dst_row = lo - h.kv_start;
      }
      ++n;
      if (o != rank) ++remote_owners;
    }
  }
  *nxfer_out = n;
  *kind_out = remote_owners == 0 ? BD_XCHG_LOCAL
              : (remote_owners == 1 && h.kv_start >= (rank - 1) * L) ? BD_XCHG_HALO : BD_XCHG_A2A;
  if (xfers && n > cap) return fail(BD_ERR_CAPACITY, "exchange needs %d transfers, capacity %d", n, cap);
  return ok();
}

namespace {

struct Built {
  std::vector<int32_t> items, segs, fwd, bwd, bwdo, rowds;
  int64_t useful = 0, fwd_tiles = 0;
  int32_t kv_rows = 0, slots = 1, qtiles = 0, nbuf = 0, C = 0, Ck = 1;
};

int32_t check_desc(const bd_plan_desc* d) {
  if (!d) return fail(BD_ERR_ARG, "plan desc is NULL");
  if (d->B <= 0 || d->S <= 0 || d->cp <= 0 || d->nchunks <= 0)
    return fail(BD_ERR_ARG, "B, S, cp and nchunks must be positive");
  if (d->S % d->cp) return fail(BD_ERR_NOT_DIVISIBLE, "S = %d not a multiple of cp = %d", d->S, d->cp);
  if (d->H <= 0 || d->Hkv <= 0 || d->H % d->Hkv)
    return fail(BD_ERR_UNSUPPORTED, "H = %d must be a positive multiple of Hkv = %d", d->H, d->Hkv);
  if (d->d != 64 && d->d != 128 && d->d != 256)
    return fail(BD_ERR_UNSUPPORTED, "head dim %d not in {64, 128, 256}", d->d);
  if (d->kv_mode != BD_KV_GATHER && d->kv_mode != BD_KV_WINDOW)
    return fail(BD_ERR_ARG, "kv_mode %d unknown", d->kv_mode);
  if (!d->cu_seqlens || !d->cu_offsets) return fail(BD_ERR_ARG, "cu_seqlens / cu_offsets NULL");
  if (d->ranks == nullptr && d->nchunks > d->cp)
    return fail(BD_ERR_ARG, "nchunks %d > cp %d without a rank list", d->nchunks, d->cp);
  for (int32_t c = 0; c < d->nchunks; ++c) {
    const int32_t r = d->ranks ? d->ranks[c] : c;
    if (r < 0 || r >= d->cp) return fail(BD_ERR_RANK, "chunk %d: rank %d outside [0, %d)", c, r, d->cp);
  }
  if (d->cu_offsets[0] < 0) return fail(BD_ERR_ARG, "cu_offsets[0] < 0");
  for (int32_t b = 0; b < d->B; ++b)
    if (d->cu_offsets[b + 1] - d->cu_offsets[b] < 1)
      return fail(BD_ERR_ARG, "sequence %d has an empty cu_seqlens array", b);
  return BD_OK;
}

int32_t build(const bd_plan_desc* d, Built* out) {
  int32_t st = check_desc(d);
  if (st) return st;
  Built& P = *out;
  const int32_t C = d->nchunks, L = d->S / d->cp, G = d->H / d->Hkv;
  P.C = C;
  P.Ck = d->kv_mode == BD_KV_GATHER ? 1 : C;
  // two query heads of a GQA group share each K/V tile; at head dim 256 one head's
  // O accumulator already takes half of TMEM, so a CTA serves a single head
  P.slots = (d->d != 256 && G % 2 == 0) ? 2 : 1;
  P.qtiles = (L + kTile - 1) / kTile;
  P.nbuf = d->B * P.Ck;
  std::vector<bd_segment_t> tmp;
  std::vector<int32_t> seq_svalid(d->B);
  for (int32_t b = 0; b < d->B; ++b) {
    const int32_t* cu = d->cu_seqlens + d->cu_offsets[b];
    const int32_t nd = d->cu_offsets[b + 1] - d->cu_offsets[b] - 1;
    for (int32_t c = 0; c < C; ++c) {
      const int32_t rank = d->ranks ? d->ranks[c] : c;
      bd_chunk_hdr h;
      st = bd_segment(cu, nd, d->S, d->cp, rank, &h, nullptr, 0);
      if (st) return fail(st, "sequence %d chunk %d: %s", b, c, bd_last_error());
      tmp.resize(std::max<int32_t>(1, h.nseg));
      st = bd_segment(cu, nd, d->S, d->cp, rank, &h, tmp.data(), h.nseg);
      if (st) return st;
      seq_svalid[b] = h.s_valid;
      int64_t useful = 0;
      for (int32_t s = 0; s < h.nseg; ++s) {
        const bd_segment_t& g = tmp[s];
        useful += int64_t(g.q_len) * g.diag_off + int64_t(g.q_len) * (g.q_len + 1) / 2;
      }
      P.useful += useful;
      const int32_t kv_base = d->kv_mode == BD_KV_GATHER ? 0 : h.kv_start;
      const int32_t item[kItemWords] = {b, c, rank, h.row_offset, h.s_valid, h.n_pad, h.kv_start,
                                        h.kv_end, int32_t(P.segs.size() / kSegWords), h.nseg,
                                        kv_base, d->kv_mode == BD_KV_GATHER ? b : b * C + c,
                                        int32_t(useful & 0x7fffffff), int32_t(useful >> 31), 0, 0};
      P.items.insert(P.items.end(), item, item + kItemWords);
      for (int32_t s = 0; s < h.nseg; ++s) {
        const bd_segment_t& g = tmp[s];
        const int32_t w[kSegWords] = {g.doc, g.q_start, g.q_len, g.k_start, g.k_len, g.diag_off};
        P.segs.insert(P.segs.end(), w, w + kSegWords);
      }
      P.kv_rows = std::max(P.kv_rows, d->kv_mode == BD_KV_GATHER ? h.s_valid : h.kv_end - h.kv_start);
      // per-row document start: segments cover the chunk's valid rows in order; an
      // item's rows take Lpad words (rows past L are invalid), so that a query
      // tile's 128 starts are one aligned 512-byte block
      {
        const size_t base = P.rowds.size();
        P.rowds.resize(base + size_t(P.qtiles) * kTile, kRowInvalid);
        for (int32_t s = 0; s < h.nseg; ++s)
          for (int32_t r = tmp[s].q_start; r < tmp[s].q_start + tmp[s].q_len; ++r)
            P.rowds[base + (r - h.row_offset)] = tmp[s].k_start;
      }
    }
  }
  // CTAs per GPU the list orders assume (a GB300 runs one CTA per SM on its 152 SMs)
  // and the band width divisor of the length-band ordering (see the backward lists)
  constexpr int64_t kOrderCtas = 152, kBandDiv = 8;
  constexpr int64_t kShortFwdUnit = 5;  // mean key tiles per forward unit at or below which bands apply
  // ---- forward work: (item, query tile, head slot group), longest first -------------
  struct FW { int32_t w[kFwdWords]; };
  std::vector<FW> fw;
  const int32_t nitems = d->B * C;
  for (int32_t it = 0; it < nitems; ++it) {
    const int32_t* I = &P.items[size_t(it) * kItemWords];
    const int32_t row0 = I[I_ROW0], svalid = I[I_SVALID], seg0 = I[I_SEG0], nseg = I[I_NSEG];
    for (int32_t t = 0; t < P.qtiles; ++t) {
      const int32_t a = row0 + t * kTile;
      const int32_t e = std::min(std::min(row0 + (t + 1) * kTile, row0 + L), svalid);
      int32_t kt_lo = 0, nt = 0;
      if (a < e) {
        int32_t ds = -1;
        for (int32_t s = 0; s < nseg; ++s) {
          const int32_t* g = &P.segs[size_t(seg0 + s) * kSegWords];
          if (a >= g[1] && a < g[1] + g[2]) { ds = g[3]; break; }
        }
        if (ds < 0) return fail(BD_ERR_PLAN, "internal: row %d has no segment", a);
        kt_lo = ds / kTile;
        nt = (e - 1) / kTile - kt_lo + 1;
      }
      for (int32_t g = 0; g < d->Hkv; ++g)
        for (int32_t p = 0; p < G / P.slots; ++p) {
          FW f = {{it, t, g * G + p * P.slots, kt_lo, nt, 0, 0, 0}};
          fw.push_back(f);
          P.fwd_tiles += nt;
        }
    }
  }
  // Longest first. When the units are short (at most 5 key tiles on average per
  // unit that has any), a K/V tile's readers are a few neighbouring query tiles, and
  // the forward streams K/V from DRAM near the bandwidth limit unless those run at
  // the same time: such lists run longest first only down to bands of similar
  // length (the backward lists' ordering, below) and in position order within a
  // band, so that neighbouring query tiles share their key tiles through L2. On
  // layouts of longer units that order measured slower than plain longest first.
  {
    int64_t total = 0, live = 0;
    for (const FW& x : fw) {
      total += x.w[F_NT];
      live += x.w[F_NT] > 0;
    }
    const int64_t band = live > 0 && total <= kShortFwdUnit * live
                             ? std::max<int64_t>(1, total / (kOrderCtas * kBandDiv))
                             : 1;
    std::stable_sort(fw.begin(), fw.end(),
                     [band](const FW& x, const FW& y) { return x.w[F_NT] / band > y.w[F_NT] / band; });
  }
  for (const FW& f : fw) P.fwd.insert(P.fwd.end(), f.w, f.w + kFwdWords);

  // ---- backward work: (K/V buffer, key tile, K/V head), most query tiles first -------
  struct BW { int32_t w[kBwdWords]; };
  const int32_t qstep = bwd_query_step(d->d);
  // query range and (query step) count of the key rows [c0, last] of sequence b over
  // chunk items [it_lo, it_hi): the rows attending to them are [c0, end of last's document)
  auto query_span = [&](int32_t b, int32_t it_lo, int32_t it_hi, int32_t c0, int32_t last, int32_t* nq,
                        int32_t* q_lo, int32_t* q_hi) {
    *nq = 0;
    *q_lo = *q_hi = c0;
    if (last < c0) return;
    const int32_t* cu = d->cu_seqlens + d->cu_offsets[b];
    const int32_t nd = d->cu_offsets[b + 1] - d->cu_offsets[b] - 1;
    const int32_t q_end = *std::upper_bound(cu + 1, cu + nd + 1, last);
    *q_hi = q_end;
    for (int32_t it = it_lo; it < it_hi; ++it) {
      const int32_t* I = &P.items[size_t(it) * kItemWords];
      const int32_t lo = std::max(c0, I[I_ROW0]), hi = std::min(q_end, I[I_ROW0] + L);
      if (lo < hi) *nq += (hi - 1 - I[I_ROW0]) / qstep - (lo - I[I_ROW0]) / qstep + 1;
    }
  };
  // CTAs claim units in list order as they finish the previous one. A list runs
  // longest first (longest-processing-time order: the last units to start are
  // short ones, so the CTAs finish together), but only down to bands of similar
  // length: within a band the units keep the order they are built in (K/V
  // buffer, key tile, K/V head), so that the CTAs working at the same time hold
  // neighbouring key tiles, whose steps read the same Q / dO tiles and add into
  // the same dQ rows through L2. A band spans 1/kBandDiv of an even share of all
  // steps over kOrderCtas CTAs (a GB300 runs one CTA per SM on its 152 SMs); the
  // finishing spread this adds is at most one band. Layouts of short documents,
  // whose units are all shorter than a band, run in position order.
  auto lpt_order = [&](std::vector<BW>& v) {
    int64_t total = 0;
    for (const BW& x : v) total += x.w[W_NQ];
    const int64_t band = std::max<int64_t>(1, total / (kOrderCtas * kBandDiv));
    std::stable_sort(v.begin(), v.end(),
                     [band](const BW& x, const BW& y) { return x.w[W_NQ] / band > y.w[W_NQ] / band; });
  };
  std::vector<BW> bw;
  for (int32_t nb = 0; nb < P.nbuf; ++nb) {
    const int32_t b = nb / P.Ck;
    const int32_t it_lo = d->kv_mode == BD_KV_GATHER ? b * C : nb;
    const int32_t it_hi = d->kv_mode == BD_KV_GATHER ? (b + 1) * C : nb + 1;
    const int32_t* I0 = &P.items[size_t(it_lo) * kItemWords];
    const int32_t kv_base = I0[I_KVBASE], svalid = I0[I_SVALID];
    const int32_t rows = d->kv_mode == BD_KV_GATHER ? d->S : I0[I_KVEND] - I0[I_KVSTART];
    const int32_t ntiles = (rows + kTile - 1) / kTile;
    for (int32_t kt = 0; kt < ntiles; ++kt) {
      const int32_t c0 = kv_base + kt * kTile;
      const int32_t last = std::min(std::min(c0 + kTile, kv_base + rows), svalid) - 1;
      int32_t nq, q_lo, q_hi;
      query_span(b, it_lo, it_hi, c0, last, &nq, &q_lo, &q_hi);
      for (int32_t g = 0; g < d->Hkv; ++g) {
        BW w = {{nb, kt * kTile, g, it_lo, it_hi, nq * G, q_lo, q_hi, c0, nb, kt * kTile, 0}};
        bw.push_back(w);
      }
    }
  }
  lpt_order(bw);
  // ---- owner-keyed backward work of a needed-only-window plan over every chunk --------
  // (sequence, tile of the global 128-row grid, K/V head): the tile lies inside the
  // rows of one chunk (L % 128 == 0) and so inside that chunk's window, from which
  // K / V are read; every chunk's query steps add into the same TMEM accumulators
  // and the sum is stored once at the owner rows.
  bool all_chunks = C == d->cp;
  for (int32_t c = 0; all_chunks && c < C; ++c)
    if (d->ranks && d->ranks[c] != c) all_chunks = false;
  if (d->kv_mode == BD_KV_WINDOW && all_chunks && L % kTile == 0) {
    std::vector<BW> bo;
    for (int32_t b = 0; b < d->B; ++b) {
      const int32_t svalid = P.items[size_t(b * C) * kItemWords + I_SVALID];
      for (int32_t kt = 0; kt < d->S / kTile; ++kt) {
        const int32_t c0 = kt * kTile, c_own = c0 / L, it_own = b * C + c_own;
        const int32_t* Io = &P.items[size_t(it_own) * kItemWords];
        const int32_t last = std::min(c0 + kTile, svalid) - 1;
        int32_t nq, q_lo, q_hi;
        query_span(b, b * C, (b + 1) * C, c0, last, &nq, &q_lo, &q_hi);
        const int32_t lrow = last >= c0 ? c0 - Io[I_KVSTART] : 0;
        for (int32_t g = 0; g < d->Hkv; ++g) {
          BW w = {{it_own, lrow, g, b * C, (b + 1) * C, nq * G, q_lo, q_hi, c0, b, c0, 0}};
          bo.push_back(w);
        }
      }
    }
    lpt_order(bo);
    for (const BW& w : bo) P.bwdo.insert(P.bwdo.end(), w.w, w.w + kBwdWords);
  }
  for (const BW& w : bw) P.bwd.insert(P.bwd.end(), w.w, w.w + kBwdWords);
  return BD_OK;
}

size_t words_of(const Built& P) {
  auto al = [](size_t x) { return (x + 3) & ~size_t(3); };  // keep 16-byte alignment per section
  return kHdrWords + al(P.items.size()) + al(P.segs.size()) + al(P.fwd.size()) + al(P.bwd.size()) +
         al(P.bwdo.size()) + al(P.rowds.size());
}

}  // namespace

extern "C" int32_t bd_plan_bytes(const bd_plan_desc* desc, size_t* bytes) {
  if (!bytes) return fail(BD_ERR_ARG, "bytes is NULL");
  Built P;
  int32_t st = build(desc, &P);
  if (st) return st;
  *bytes = words_of(P) * sizeof(int32_t);
  return ok();
}

extern "C" int32_t bd_plan_build(const bd_plan_desc* d, void* blob, size_t blob_bytes) {
  if (!blob) return fail(BD_ERR_ARG, "blob is NULL");
  if (reinterpret_cast<uintptr_t>(blob) % 16) return fail(BD_ERR_ALIGN, "blob not 16-byte aligned");
  Built P;
  int32_t st = build(d, &P);
  if (st) return st;
  const size_t words = words_of(P);
  if (blob_bytes < words * sizeof(int32_t))
    return fail(BD_ERR_CAPACITY, "plan needs %zu bytes, got %zu", words * sizeof(int32_t), blob_bytes);
  if (words > size_t(INT32_MAX)) return fail(BD_ERR_CAPACITY, "plan too large");
  int32_t* w = static_cast<int32_t*>(blob);
  std::memset(w, 0, words * sizeof(int32_t));
  auto al = [](size_t x) { return int32_t((x + 3) & ~size_t(3)); };
  int32_t off = kHdrWords;
  const float scale = 1.0f / std::sqrt(float(d->d));
  int32_t scale_bits;
  std::memcpy(&scale_bits, &scale, 4);
  w[H_MAGIC] = kPlanMagic; w[H_VERSION] = kPlanVersion; w[H_WORDS] = int32_t(words);
  w[H_B] = d->B; w[H_S] = d->S; w[H_CP] = d->cp; w[H_C] = d->nchunks; w[H_L] = d->S / d->cp;
  w[H_H] = d->H; w[H_HKV] = d->Hkv; w[H_D] = d->d; w[H_KVMODE] = d->kv_mode; w[H_G] = d->H / d->Hkv;
  w[H_NITEMS] = d->B * d->nchunks;
  w[H_OFF_ITEMS] = off; std::copy(P.items.begin(), P.items.end(), w + off); off += al(P.items.size());
  w[H_OFF_SEGS] = off; w[H_NSEGS] = int32_t(P.segs.size() / kSegWords);
  std::copy(P.segs.begin(), P.segs.end(), w + off); off += al(P.segs.size());
  w[H_OFF_FWD] = off; w[H_NFWD] = int32_t(P.fwd.size() / kFwdWords);
  std::copy(P.fwd.begin(), P.fwd.end(), w + off); off += al(P.fwd.size());
  w[H_OFF_BWD] = off; w[H_NBWD] = int32_t(P.bwd.size() / kBwdWords);
  std::copy(P.bwd.begin(), P.bwd.end(), w + off); off += al(P.bwd.size());
  w[H_OFF_BWDO] = off; w[H_NBWDO] = int32_t(P.bwdo.size() / kBwdWords);
  std::copy(P.bwdo.begin(), P.bwdo.end(), w + off); off += al(P.bwdo.size());
  w[H_OFF_ROWDS] = off;
  std::copy(P.rowds.begin(), P.rowds.end(), w + off); off += al(P.rowds.size());
  w[H_SCALE_BITS] = scale_bits; w[H_KV_ROWS] = P.kv_rows; w[H_CK] = P.Ck; w[H_SLOTS] = P.slots;
  w[H_QTILES] = P.qtiles;
  w[H_USEFUL_LO] = int32_t(P.useful & 0x7fffffff); w[H_USEFUL_HI] = int32_t(P.useful >> 31);
  w[H_NBUF] = P.nbuf;
  w[H_FWD_TILES_LO] = int32_t(P.fwd_tiles & 0x7fffffff); w[H_FWD_TILES_HI] = int32_t(P.fwd_tiles >> 31);
  return ok();
}

extern "C" int32_t bd_plan_chunk(const void* plan_host, int32_t item, bd_chunk_hdr* hdr,
                                 bd_segment_t* segs, int32_t seg_capacity) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!hdr) return fail(BD_ERR_ARG, "hdr is NULL");
  if (item < 0 || item >= pv.hdr(H_NITEMS)) return fail(BD_ERR_ARG, "item %d out of range", item);
  const int32_t* I = pv.item(item);
  hdr->S = pv.hdr(H_S); hdr->cp = pv.hdr(H_CP); hdr->rank = I[I_RANK]; hdr->L = pv.hdr(H_L);
  hdr->row_offset = I[I_ROW0]; hdr->s_valid = I[I_SVALID]; hdr->n_pad = I[I_NPAD];
  hdr->kv_start = I[I_KVSTART]; hdr->kv_end = I[I_KVEND]; hdr->nseg = I[I_NSEG];
  if (segs) {
    if (seg_capacity < I[I_NSEG]) return fail(BD_ERR_CAPACITY, "need %d segments", I[I_NSEG]);
    for (int32_t s = 0; s < I[I_NSEG]; ++s) {
      const int32_t* g = pv.seg(I[I_SEG0] + s);
      segs[s].doc = g[0]; segs[s].q_start = g[1]; segs[s].q_len = g[2];
      segs[s].k_start = g[3]; segs[s].k_len = g[4]; segs[s].diag_off = g[5];
    }
  }
  return ok();
}

extern "C" int32_t bd_plan_set_dropout(void* plan_host, double p, uint64_t seed) {
  PlanView pv;
  int32_t st = view_plan(plan_host, &pv);
  if (st) return st;
  if (!(p >= 0.0 && p < 1.0)) return fail(BD_ERR_ARG, "dropout probability %g not in [0, 1)", p);
  const double t = std::floor(p * 4294967296.0 + 0.5);
  const uint32_t thresh = t >= 4294967295.0 ? 0xFFFFFFFFu : uint32_t(t);
  const float scale = float(1.0 / (1.0 - p));
  int32_t* h = static_cast<int32_t*>(plan_host);
  int32_t sbits;
  memcpy(&sbits, &scale, 4);
  h[H_DROP_THRESH] = int32_t(thresh);
  h[H_DROP_SCALE_BITS] = sbits;
  h[H_DROP_SEED_LO] = int32_t(uint32_t(seed & 0xFFFFFFFFu));
  h[H_DROP_SEED_HI] = int32_t(uint32_t(seed >> 32));
  return ok();
}

extern "C" int64_t bd_plan_useful_pairs(const void* plan_host) {
  PlanView pv;
  if (view_plan(plan_host, &pv)) return -1;
  return (int64_t(pv.hdr(H_USEFUL_HI)) << 31) | int64_t(pv.hdr(H_USEFUL_LO));
}
