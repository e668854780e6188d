/* A C99 consumer of include/bd_attn.h: compiled and run by tests/test_c_consumer.py
 * (host calls only, no GPU). It prints the segmentation of the 3-document layout
 * cu_seqlens = [0, 200, 350, 512], S = 512, cp = 2 (the hand-derived fixture in
 * tests/golden/segment_tiny_3docs.txt), the same metadata read back from a plan
 * built through bd_plan_desc, the sizes of the ABI structs, and the statuses of
 * a few rejected calls. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "bd_attn.h"

static int check(int32_t st, const char* what) {
  if (st != BD_OK) {
    printf("error %s %d %s\n", what, (int)st, bd_last_error());
    return 1;
  }
  return 0;
}

int main(void) {
  const int32_t cu[4] = {0, 200, 350, 512};
  const int32_t S = 512, cp = 2;
  int32_t r, i;
  printf("layout %d %d", (int)S, (int)cp);
  for (i = 0; i < 4; ++i) printf(" %d", (int)cu[i]);
  printf("\n");
  for (r = 0; r < cp; ++r) {
    bd_chunk_hdr h;
    bd_segment_t segs[8];
    if (check(bd_segment(cu, 3, S, cp, r, &h, segs, 8), "bd_segment")) return 1;
    printf("chunk %d %d %d %d %d %d %d\n", (int)h.rank, (int)h.row_offset, (int)h.s_valid, (int)h.n_pad,
           (int)h.kv_start, (int)h.kv_end, (int)h.nseg);
    for (i = 0; i < h.nseg; ++i)
      printf("seg %d %d %d %d %d %d\n", (int)segs[i].doc, (int)segs[i].q_start, (int)segs[i].q_len,
             (int)segs[i].k_start, (int)segs[i].k_len, (int)segs[i].diag_off);
  }
  /* the same chunks through a plan over both chunks (the batched form) */
  {
    const int32_t offs[2] = {0, 4};
    bd_plan_desc d;
    size_t bytes = 0;
    unsigned char* raw;
    void* blob;
    memset(&d, 0, sizeof d);
    d.B = 1; d.S = S; d.cp = cp; d.nchunks = cp; d.ranks = NULL;
    d.H = 4; d.Hkv = 4; d.d = 64; d.kv_mode = BD_KV_WINDOW;
    d.cu_seqlens = cu; d.cu_offsets = offs;
    if (check(bd_plan_bytes(&d, &bytes), "bd_plan_bytes")) return 1;
    raw = (unsigned char*)malloc(bytes + 64); /* the blob must be 16-byte aligned */
    if (!raw) return 1;
    blob = raw + ((64 - (size_t)raw % 64) % 64);
    if (check(bd_plan_build(&d, blob, bytes), "bd_plan_build")) return 1;
    for (r = 0; r < cp; ++r) {
      bd_chunk_hdr h;
      bd_segment_t segs[8];
      if (check(bd_plan_chunk(blob, r, &h, segs, 8), "bd_plan_chunk")) return 1;
      printf("plan_chunk %d %d %d %d %d %d %d\n", (int)h.rank, (int)h.row_offset, (int)h.s_valid, (int)h.n_pad,
             (int)h.kv_start, (int)h.kv_end, (int)h.nseg);
    }
    printf("useful %lld\n", (long long)bd_plan_useful_pairs(blob));
    free(raw);
  }
  {
    int32_t ids[6] = {0, 0, 1, 1, 1, -1}, out[4], nd = 0;
    if (check(bd_doc_ids_to_cu(ids, 6, out, 4, &nd), "bd_doc_ids_to_cu")) return 1;
    printf("doc_ids_to_cu %d %d %d %d\n", (int)nd, (int)out[0], (int)out[1], (int)out[2]);
  }
  {
    bd_chunk_hdr h;
    const int32_t bad[3] = {0, 300, 200};
    printf("reject %d %d %d\n", (int)bd_segment(bad, 2, S, cp, 0, &h, NULL, 0), (int)bd_segment(cu, 3, 513, cp, 0, &h, NULL, 0),
           (int)bd_segment(cu, 3, S, cp, 2, &h, NULL, 0));
  }
  printf("sizeof %u %u %u %u %u %u\n", (unsigned)sizeof(bd_segment_t), (unsigned)sizeof(bd_chunk_hdr),
         (unsigned)sizeof(bd_plan_desc), (unsigned)sizeof(bd_tensor), (unsigned)sizeof(bd_rowstat),
         (unsigned)sizeof(bd_xfer_t));
  printf("version %d\n", (int)bd_version());
  return 0;
}
