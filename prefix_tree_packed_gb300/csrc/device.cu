// Per-device facts and tensor maps the launchers need.
#include <cudaTypedefs.h>

#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"

namespace tree {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kSMs;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kSMs;
    cached[dev] = n;
  }
  return cached[dev];
}

int set_max_dynamic_smem(const void *fn, int bytes, const char *who) {
  // a kernel attribute belongs to one device: a process that launches on a
  // second device sets it again there
  static std::mutex mu;
  static std::set<std::pair<int, const void *>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, fn})) return TREE_OK;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  done.insert({dev, fn});
  return TREE_OK;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

int make_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, const char *who, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return fail(TREE_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", who);
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TREE_ERR_CUDA, "%s: tensor map encode failed (%d)", who, (int)r);
  return TREE_OK;
}

}  // namespace tree
