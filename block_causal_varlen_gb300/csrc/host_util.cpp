#include "host_util.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace bd {

int32_t cuda_fail(cudaError_t e, const char* what) {
  return fail(BD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int32_t check_tensor(const bd_tensor* t, const char* name, int elem_bytes, int64_t B, int64_t C, int64_t H,
                     bool need_tma) {
  if (!t || !t->ptr) return fail(BD_ERR_ARG, "%s: NULL tensor or pointer", name);
  if (t->rows <= 0) return fail(BD_ERR_ARG, "%s: rows must be positive", name);
  if (reinterpret_cast<uintptr_t>(t->ptr) % 16) return fail(BD_ERR_ALIGN, "%s: base not 16-byte aligned", name);
  const int64_t st[4] = {t->stride_b, t->stride_c, t->stride_row, t->stride_head};
  const int64_t ext[4] = {B, C, t->rows, H};
  const char* nm[4] = {"b", "c", "row", "head"};
  for (int i = 0; i < 4; ++i) {
    if (ext[i] <= 1) continue;
    if (st[i] <= 0) return fail(BD_ERR_ALIGN, "%s: stride_%s must be positive", name, nm[i]);
    if ((st[i] * elem_bytes) % 16)
      return fail(BD_ERR_ALIGN, "%s: stride_%s (%lld elements) is not a multiple of 16 bytes", name, nm[i],
                  (long long)st[i]);
    if (need_tma && st[i] * elem_bytes >= (int64_t(1) << 40))
      return fail(BD_ERR_ALIGN, "%s: stride_%s too large for TMA", name, nm[i]);
  }
  return BD_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static int32_t make_tmap(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                         const char* name, int esize, CUtensorMapDataType dtype, cuuint32_t box0,
                         CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B, cuuint32_t box_rows = 128,
                         cuuint32_t box_heads = 1) {
  auto fn = encode_fn();
  if (!fn) return fail(BD_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
  auto fix = [esize](int64_t stride_elems, int64_t ext, int64_t fallback) {
    return ext <= 1 ? fallback : stride_elems * esize;
  };
  const int64_t sh = fix(t->stride_head, heads, d * esize);
  const int64_t sr = fix(t->stride_row, t->rows, sh * heads);
  const int64_t sc = fix(t->stride_c, C, sr * t->rows);
  const int64_t sb = fix(t->stride_b, B, sc * C);
  cuuint64_t dims[5] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(t->rows), cuuint64_t(C), cuuint64_t(B)};
  cuuint64_t strides[4] = {cuuint64_t(sh), cuuint64_t(sr), cuuint64_t(sc), cuuint64_t(sb)};
  cuuint32_t box[5] = {box0, box_heads, box_rows, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dtype, 5, t->ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(BD_ERR_ALIGN, "%s: cuTensorMapEncodeTiled failed (%d)", name, int(r));
  return BD_OK;
}

int32_t make_tmap_f32_reduce(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                             const char* name, int box_cols, int box_rows) {
  if (box_cols != 16 && box_cols != 32 && box_cols != 128)
    return fail(BD_ERR_ARG, "%s: reduce box of %d columns", name, box_cols);
  // 16 / 32 columns: 64- / 128-byte swizzled rows; 128 columns: 512-byte rows, unswizzled
  const CUtensorMapSwizzle swz = box_cols == 32    ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : box_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
  return make_tmap(map, t, B, C, heads, d, name, 4, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cuuint32_t(box_cols), swz,
                   cuuint32_t(box_rows));
}

int32_t make_tmap_bf16(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                       const char* name, int box_rows) {
  return make_tmap(map, t, B, C, heads, d, name, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                   cuuint32_t(box_rows));
}

int32_t make_tmap_rows_bf16(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                            const char* name, int box_heads, int box_rows) {
  if (d > 256 || box_heads < 1 || box_heads > 256 || box_rows < 1 || box_rows > 256)
    return fail(BD_ERR_ARG, "%s: row box of %lld columns x %d heads x %d rows", name, (long long)d, box_heads,
                box_rows);
  return make_tmap(map, t, B, C, heads, d, name, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(d),
                   CU_TENSOR_MAP_SWIZZLE_NONE, cuuint32_t(box_rows), cuuint32_t(box_heads));
}

int32_t sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static int cache[64] = {0};
  if (dev < 64 && cache[dev]) {
    *out = cache[dev];
    return BD_OK;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if (dev < 64) cache[dev] = n;
  *out = n;
  return BD_OK;
}

}  // namespace bd
