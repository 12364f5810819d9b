// KV-cache write through a slot mapping, and the page gather used to check page indexing.
//
// Both are pure copies (bit-exact) bound by HBM bandwidth: 16-byte vector loads and stores of
// 16-byte chunks of token rows (rows of num_kv_heads*head_dim*2 bytes).
#include "common.cuh"

namespace {

using namespace pkv;

// Two 16-byte chunks of token rows per thread and loop step, K and V: every load of a step (the
// slot, two K chunks, two V chunks) is issued before any of them is used, so a thread keeps 64
// bytes of new K/V in flight and the step costs one memory latency, not two (the slot check
// would otherwise hold back the K/V loads).  The new rows are read once: non-caching loads.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(256) kv_append_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int64_t* __restrict__ slots, int32_t num_tokens,
    int32_t chunks_per_row, int64_t num_slots, uint32_t* err_word) {
  const int64_t total = (int64_t)num_tokens * chunks_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    const int64_t i1 = i0 + stride;
    const bool has1 = i1 < total;
    const int64_t t0 = i0 / chunks_per_row, t1 = has1 ? i1 / chunks_per_row : t0;
    const uint4 k0 = ld_stream(k_new + i0), v0 = ld_stream(v_new + i0);
    uint4 k1 = make_uint4(0u, 0u, 0u, 0u), v1 = k1;
    if (has1) {
      k1 = ld_stream(k_new + i1);
      v1 = ld_stream(v_new + i1);
    }
    const int64_t s0 = __ldg(slots + t0), s1 = __ldg(slots + t1);
    const int64_t c0 = i0 - t0 * chunks_per_row, c1 = i1 - t1 * chunks_per_row;
    // a negative slot is a padding token; one past the pool is reported (once per row)
    if (s0 >= num_slots && c0 == 0) report(err_word, PKV_DEVERR_SLOT_OOB);
    if (has1 && s1 >= num_slots && c1 == 0) report(err_word, PKV_DEVERR_SLOT_OOB);
    if (s0 >= 0 && s0 < num_slots) {
      k_pool[s0 * chunks_per_row + c0] = k0;
      v_pool[s0 * chunks_per_row + c0] = v0;
    }
    if (has1 && s1 >= 0 && s1 < num_slots) {
      k_pool[s1 * chunks_per_row + c1] = k1;
      v_pool[s1 * chunks_per_row + c1] = v1;
    }
  }
}

// Block (x, b): request b's rows, split over gridDim.x blocks.  The output offset of request b is
// the sum of the earlier lengths, recomputed by each block (a debug op: B is small).
__global__ void __launch_bounds__(256) paged_gather_kernel(
    const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
    const int32_t* __restrict__ kv_indptr, const int32_t* __restrict__ kv_indices,
    const int32_t* __restrict__ kv_lens, int32_t page_size, int64_t num_pages,
    int32_t chunks_per_row, uint4* __restrict__ k_out, uint4* __restrict__ v_out,
    uint32_t* err_word) {
  const int b = blockIdx.y;
  __shared__ int64_t s_offset;
  if (threadIdx.x < 32) {
    int64_t acc = 0;
    for (int i = threadIdx.x; i < b; i += 32) acc += __ldg(kv_lens + i);
    acc = warp_sum(acc);
    if (threadIdx.x == 0) s_offset = acc;
  }
  __syncthreads();
  const int64_t out0 = s_offset;
  const int32_t L = __ldg(kv_lens + b);
  const int32_t p0 = __ldg(kv_indptr + b), p1 = __ldg(kv_indptr + b + 1);
  const int64_t total = (int64_t)L * chunks_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / chunks_per_row;
    const int64_t c = i - j * chunks_per_row;
    const int64_t pslot = p0 + j / page_size;
    if (pslot >= p1) {
      if (c == 0) report(err_word, PKV_DEVERR_LENGTH);
      continue;
    }
    const int64_t page = __ldg(kv_indices + pslot);
    if (page < 0 || page >= num_pages) {
      if (c == 0) report(err_word, PKV_DEVERR_PAGE_OOB);
      continue;
    }
    const int64_t src = (page * page_size + j % page_size) * chunks_per_row + c;
    k_out[(out0 + j) * chunks_per_row + c] = __ldg(k_pool + src);
    v_out[(out0 + j) * chunks_per_row + c] = __ldg(v_pool + src);
  }
}

}  // namespace

extern "C" {

pkv_status pkv_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int32_t num_tokens, uint32_t* err_word,
                         void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_kv_append");
  if (!pkv_host::valid_pool(pool) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!pkv_host::aligned16(k_new) || !pkv_host::aligned16(v_new)) return PKV_ERR_INVALID_ARG;
  const int64_t row_bytes = (int64_t)pool->num_kv_heads * pool->head_dim * 2;
  const int32_t chunks = (int32_t)(row_bytes / 16);
  const int64_t total = (int64_t)num_tokens * chunks;
  const int threads = 256;
  int64_t blocks = (total + 2 * threads - 1) / (2 * threads);  // two chunks per thread and step
  const int64_t cap = (int64_t)pkv_host::sm_count() * 8;
  if (cap > 0 && blocks > cap) blocks = cap;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      (uint4*)pool->k, (uint4*)pool->v, (const uint4*)k_new, (const uint4*)v_new, slot_mapping,
      num_tokens, chunks, pool->num_pages * pool->page_size, err_word);
  return pkv_host::launch_status();
}

pkv_status pkv_paged_gather(const pkv_pool* pool, const int32_t* kv_indptr,
                            const int32_t* kv_indices, const int32_t* kv_lens, int32_t batch_size,
                            void* k_out, void* v_out, uint32_t* err_word, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_gather");
  if (!pkv_host::valid_pool(pool) || batch_size < 0) return PKV_ERR_INVALID_ARG;
  if (batch_size == 0) return PKV_OK;
  if (!kv_indptr || !kv_indices || !kv_lens || !k_out || !v_out) return PKV_ERR_INVALID_ARG;
  if (!pkv_host::aligned16(k_out) || !pkv_host::aligned16(v_out)) return PKV_ERR_INVALID_ARG;
  if (batch_size > 65535) return PKV_ERR_UNSUPPORTED;
  const int32_t chunks = (int32_t)((int64_t)pool->num_kv_heads * pool->head_dim * 2 / 16);
  dim3 grid(8, batch_size);
  paged_gather_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
      (const uint4*)pool->k, (const uint4*)pool->v, kv_indptr, kv_indices, kv_lens,
      pool->page_size, pool->num_pages, chunks, (uint4*)k_out, (uint4*)v_out, err_word);
  return pkv_host::launch_status();
}

}  // extern "C"
