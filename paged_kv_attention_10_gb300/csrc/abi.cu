// C-ABI plumbing: status strings, version, host-side argument checks and device properties.
#include <cudaTypedefs.h>

#include <atomic>

#include "tc05.cuh"

namespace pkv_host {

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

int sm_count() {
  static std::atomic<int> cache[64];
  int d = current_device();
  if (d < 0) return 0;
  if (d < 64) {
    int c = cache[d].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
  if (d < 64) cache[d].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

bool valid_pool(const pkv_pool* p) {
  if (!p || !p->k || !p->v) return false;
  if (p->num_pages <= 0 || p->page_size <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0) return false;
  if ((p->head_dim % 8) != 0) return false;
  if (!aligned16(p->k) || !aligned16(p->v)) return false;
  return true;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load();
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      fn.store(f);
    }
  }
  return f;
}
}  // namespace

bool encode_tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv_host

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_WORKSPACE: return "workspace too small";
    case PKV_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int32_t pkv_version(void) { return 100; }  // 0.1.0

}  // extern "C"

namespace {

// One thread waits on an mbarrier that nothing arrives on, with the same bounded wait the
// kernels use, and reports the timeout the way they do.
__global__ void bounded_wait_selftest_kernel(uint32_t* err_word) {
  __shared__ uint64_t bar;
  pkv::mbar_init(&bar, 1);
  pkv::fence_mbar_init();
  if (!pkv::mbar_wait(&bar, 0)) pkv::report(err_word, PKV_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" {

pkv_status pkv_selftest_bounded_wait(uint32_t* err_word, void* stream) {
  if (!err_word) return PKV_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(err_word);
  return pkv_host::launch_status();
}

}  // extern "C"
