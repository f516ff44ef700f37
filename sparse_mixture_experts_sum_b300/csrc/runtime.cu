// Host runtime helpers: the driver's tensor-map encoder (looked up once
// through the runtime, so the library does not link libcuda directly) and
// per-device SM counts.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool make_tma_2d_bf16(CUtensorMap* map, const void* base, long long inner, long long rows, int box_inner,
                      int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || inner <= 0 || rows <= 0) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((inner * 2) % 16)) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
// Zero two word ranges in one small launch (the error word and a counter
// array, typically); a kernel on the compute stream rather than a memset.
__global__ void zero_words_kernel(uint32_t* __restrict__ a, long long na, uint32_t* __restrict__ b, long long nb) {
  pdl_entry();
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (i < na) a[i] = 0u;
    else b[i - na] = 0u;
  }
}
}  // namespace

moe_status launch_zero(void* a, size_t a_bytes, void* b, size_t b_bytes, cudaStream_t stream) {
  const long long na = a ? static_cast<long long>(a_bytes / 4) : 0;
  const long long nb = b ? static_cast<long long>(b_bytes / 4) : 0;
  if (na + nb == 0) return MOE_OK;
  long long blocks = (na + nb + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  launch_pdl(zero_words_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, static_cast<uint32_t*>(a),
             na, static_cast<uint32_t*>(b), nb);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int device_sm_count(int dev) {
  static DeviceOnce once;
  static int cache[64] = {0};
  const moe_status s = once.run(dev, [&] {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return MOE_ERR_CUDA;
    cache[dev] = v;
    return MOE_OK;
  });
  return s == MOE_OK ? cache[dev] : 0;
}

// Self-test of the bounded-wait path: one thread waits on a shared-memory
// barrier that expects one arrival and gets none.  The wait gives up after
// kWaitLimitNs and records kErrSelfTest in the error word; the kernel then
// returns normally, so the context stays usable.
__global__ void selftest_wait_kernel(int* err) {
  pdl_entry();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0)) record_error(err, kErrSelfTest);
}

moe_status launch_selftest_wait(int* err, cudaStream_t stream) {
  moe_status s = launch_zero(err, sizeof(int), nullptr, 0, stream);
  if (s != MOE_OK) return s;
  launch_pdl(selftest_wait_kernel, dim3(1), dim3(32), 0, stream, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
