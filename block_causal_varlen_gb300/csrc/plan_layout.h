// Layout of the plan blob that bd_plan_build writes on the host and the
// kernels read from device memory. All fields are int32; offsets count int32
// words from the start of the blob.
#pragma once
#include <stdint.h>

namespace bd {

constexpr int32_t kPlanMagic = 0x54414442;  // "BDAT"
constexpr int32_t kPlanVersion = 1;
constexpr int kTile = 128;                  // rows per query tile and per key tile

// header words
enum : int {
  H_MAGIC = 0, H_VERSION, H_WORDS, H_B, H_S, H_CP, H_C, H_L, H_H, H_HKV, H_D,
  H_KVMODE, H_G, H_NITEMS, H_OFF_ITEMS, H_OFF_SEGS, H_NSEGS, H_OFF_FWD, H_NFWD,
  H_OFF_BWD, H_NBWD, H_SCALE_BITS, H_KV_ROWS, H_CK, H_SLOTS, H_QTILES,
  H_USEFUL_LO, H_USEFUL_HI, H_NBUF, H_FWD_TILES_LO, H_FWD_TILES_HI,
  H_OFF_ROWDS,          // int32 [nitems][Lpad]: global start row of each chunk row's
                        // document, kRowInvalid for padding rows
  H_DROP_THRESH,        // attention dropout: keep iff Philox word >= this (uint32; 0 = off)
  H_DROP_SCALE_BITS,    // 1 / (1 - p) as float bits
  H_DROP_SEED_LO,       // Philox key words
  H_DROP_SEED_HI,
  H_OFF_BWDO,           // backward work units keyed by owner rows (BD_KV_WINDOW plans
  H_NBWDO,              // of every chunk in order with L % 128 == 0; else 0 units)
  H_FWD_SLOTS = 38,     // kFwdCounterSlots (claim, done) pairs of forward work-unit
                        // counters, one pair per launch in flight (0 between launches)
  H_STATUS = 56,        // written by kernels: 0 = ok, else a device failure code
  H_STATUS_DETAIL = 57, // where it happened: 1 forward, 2 backward main (either head dim),
                        // 4 backward statistics, 99 the bounded-wait self test
  kHdrWords = 64
};

// chunk item words (item = b * C + c)
enum : int {
  I_B = 0, I_C, I_RANK, I_ROW0, I_SVALID, I_NPAD, I_KVSTART, I_KVEND, I_SEG0, I_NSEG,
  I_KVBASE,   // global row held by row 0 of this item's K/V buffer
  I_KVBUF,    // K/V buffer index: b (GATHER) or b*C + c (WINDOW)
  I_USEFUL_LO, I_USEFUL_HI, I_RESERVED0, I_RESERVED1,
  kItemWords = 16
};

constexpr int32_t kRowInvalid = 0x7fffffff;

constexpr int kSegWords = 6;  // doc, q_start, q_len, k_start, k_len, diag_off

// forward work unit: one 128-row query tile of one item for `slots` query
// heads of one K/V head group, visiting key tiles [kt_lo, kt_lo + nt) of
// the global 128-row grid.
enum : int { F_ITEM = 0, F_QTILE, F_H0, F_KTLO, F_NT, F_PAD0, F_PAD1, F_PAD2, kFwdWords = 8 };

// backward work unit: one 128-row tile of keys of one K/V head. K and V are
// read from K/V buffer W_BUF at buffer rows [W_LROW, W_LROW + 128); the tile's
// first key is global row W_KEY0; its dK / dV rows leave for output buffer
// W_OBUF at rows [W_OROW, W_OROW + 128). The unit visits the query tiles of
// chunk items [item_lo, item_hi) that hold global rows in [q_lo, q_hi): the
// rows that attend to at least one key of the tile (q_lo = q_hi when none).
// nq counts (query step, query head) pairs; a query step is bwd_query_step(d)
// rows of one chunk.
// The plan's main list has one unit per (K/V buffer, 128-row tile of that
// buffer, K/V head), output = the same buffer and rows. The owner list of a
// needed-only-window plan has one unit per (sequence, 128-row tile of the
// global row grid, K/V head): it reads the tile from the window of the chunk
// that owns those rows and sums every chunk's contribution into the owner
// rows of a [B, 1, S, Hkv, d] output.
enum : int {
  W_BUF = 0, W_LROW, W_G, W_ITEM_LO, W_ITEM_HI, W_NQ, W_QLO, W_QHI, W_KEY0, W_OBUF, W_OROW, W_PAD0,
  kBwdWords = 12
};

// Query rows per backward step: 128, and 64 at head dim 256, where a 128-row Q
// tile and dO tile (64 KB each) would not fit in shared memory next to the
// resident K and V tiles.
constexpr int bwd_query_step(int d) { return d == 256 ? 64 : kTile; }

// device failure codes stored at H_STATUS
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_SMEM_ALIGN = 2 };

// Forward launches take their work-unit counters from one of these slots in the
// device plan, in turn (launch k uses slot k mod kFwdCounterSlots), so that up to
// this many forward launches sharing one device plan may run at the same time.
constexpr int kFwdCounterSlots = 8;
static_assert(H_FWD_SLOTS + 2 * kFwdCounterSlots <= H_STATUS, "forward counter slots overlap the status words");

}  // namespace bd
