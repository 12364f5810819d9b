// C-ABI plumbing: status strings, version, host-side argument checks and device properties.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <utility>
#include <vector>

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

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

void* driver_entry(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return p;
}
}  // namespace

unsigned long long current_context_id() {
  static std::atomic<CtxGetCurrentFn> get_cur{nullptr};
  static std::atomic<CtxGetIdFn> get_id{nullptr};
  CtxGetCurrentFn fc = get_cur.load();
  CtxGetIdFn fi = get_id.load();
  if (!fc || !fi) {
    fc = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent", 4000));
    fi = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId", 12000));
    if (!fc || !fi) return 0;
    get_cur.store(fc);
    get_id.store(fi);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fc(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (fi(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

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

pkv_status pkv_validate_page_table(const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* kv_lens, int32_t batch_size, int64_t num_pages,
                                   int32_t page_size, int32_t min_len, int32_t* bad_request) {
  if (bad_request) *bad_request = -1;
  if (batch_size < 0 || num_pages < 0 || page_size <= 0 || min_len < 0) return PKV_ERR_INVALID_ARG;
  if (batch_size == 0) return PKV_OK;
  if (!kv_indptr || !kv_lens || (!kv_indices && kv_indptr[batch_size] > 0)) return PKV_ERR_INVALID_ARG;
  auto bad = [&](int32_t b) {
    if (bad_request) *bad_request = b;
    return PKV_ERR_INVALID_ARG;
  };
  if (kv_indptr[0] != 0) return bad(0);
  for (int32_t b = 0; b < batch_size; ++b) {
    const int64_t lo = kv_indptr[b], hi = kv_indptr[b + 1];
    if (hi < lo) return bad(b);
    const int64_t len = kv_lens[b];
    if (len < min_len || len > (hi - lo) * (int64_t)page_size) return bad(b);
    for (int64_t k = lo; k < hi; ++k)
      if (kv_indices[k] < 0 || kv_indices[k] >= num_pages) return bad(b);
  }
  return PKV_OK;
}

pkv_status pkv_validate_slots(const int64_t* slot_mapping, int32_t num_tokens, int64_t num_slots,
                              int32_t* bad_token) {
  if (bad_token) *bad_token = -1;
  if (num_tokens < 0 || num_slots < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!slot_mapping) return PKV_ERR_INVALID_ARG;
  std::vector<std::pair<int64_t, int32_t>> used;  // (slot, token) of every non-padding token
  used.reserve((size_t)num_tokens);
  for (int32_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;  // padding
    if (s >= num_slots) {
      if (bad_token) *bad_token = t;
      return PKV_ERR_INVALID_ARG;
    }
    used.emplace_back(s, t);
  }
  std::sort(used.begin(), used.end());
  int32_t first_dup = -1;  // the later token of the earliest duplicated pair, in token order
  for (size_t i = 1; i < used.size(); ++i)
    if (used[i].first == used[i - 1].first && (first_dup < 0 || used[i].second < first_dup))
      first_dup = used[i].second;
  if (first_dup >= 0) {
    if (bad_token) *bad_token = first_dup;
    return PKV_ERR_INVALID_ARG;
  }
  return PKV_OK;
}

pkv_status pkv_selftest_bounded_wait(uint32_t* err_word, void* stream) {
  if (!err_word) return PKV_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(err_word);
  return pkv_host::launch_status();
}

}  // extern "C"
