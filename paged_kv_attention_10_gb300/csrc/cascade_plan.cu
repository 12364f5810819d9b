// Host plan of a shared-prefix (cascade) decode: integer bookkeeping over the batch's page lists,
// no attention arithmetic.  Requests of a radix-cache group share the physical pages of a prefix
// (mini-sglang README, "KVcache Management": Radix Attention); the plan lists the parts that
// attend a group's queries to chunks of the shared pages (pkv_shared_prefix_attention) and the
// page list of each request's own positions (a decode), whose partial states
// pkv_merge_states_bf16 then merges.  It is the "plan" half of the plan/run split the handbook
// describes for FlashInfer ("mini-sglang from Scratch", "What you will be able to do").
#include <algorithm>
#include <cstdint>
#include <vector>

#include "common.cuh"

namespace {

constexpr int kTileRows = 128;  // query rows (token, group head) per tile of the shared-prefix kernel

struct KeptGroup {
  int32_t first, count, shared_pages;
};

}  // namespace

extern "C" pkv_status pkv_plan_shared_prefix(
    const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_lens, int32_t batch_size,
    const int32_t* group_first, const int32_t* group_count, int32_t num_groups, int32_t page_size,
    int32_t num_kv_heads, int32_t group_size, int32_t num_sms, int32_t ctas_per_sm,
    int32_t min_chunk_tokens, pkv_cascade_sizes* sizes, int32_t* shared_tokens, int32_t* part_q_start,
    int32_t* part_q_len, int32_t* part_o_start, int32_t* part_kv_indptr, int32_t* part_kv_indices,
    int32_t* part_kv_lens, int32_t* suffix_kv_indptr, int32_t* suffix_kv_indices,
    int32_t* suffix_kv_lens, int32_t parts_capacity, int32_t indices_capacity) {
  const int32_t B = batch_size;
  if (!sizes || B <= 0 || num_groups < 0 || page_size <= 0 || num_kv_heads <= 0 || group_size < 1 ||
      group_size > 16 || num_sms <= 0 || ctas_per_sm <= 0 || min_chunk_tokens < 0)
    return PKV_ERR_INVALID_ARG;
  if (!kv_indptr || !kv_lens || (num_groups > 0 && (!group_first || !group_count)))
    return PKV_ERR_INVALID_ARG;
  if (kv_indptr[0] != 0) return PKV_ERR_INVALID_ARG;
  for (int32_t r = 0; r < B; ++r)
    if (kv_indptr[r + 1] < kv_indptr[r]) return PKV_ERR_INVALID_ARG;
  if (kv_indptr[B] > 0 && !kv_indices) return PKV_ERR_INVALID_ARG;
  const int64_t ps = page_size;
  const int32_t tpt = kTileRows / group_size;  // tokens per Q tile

  // groups: the longest common leading run of page ids, cut so that every member keeps at least
  // one position of its own
  std::vector<int32_t> owner((size_t)B, -1);
  std::vector<KeptGroup> kept;
  for (int32_t g = 0; g < num_groups; ++g) {
    const int32_t first = group_first[g], count = group_count[g];
    if (count < 1 || first < 0 || first > B - count) return PKV_ERR_INVALID_ARG;
    for (int32_t r = first; r < first + count; ++r)
      if (owner[r] >= 0 || owner[r] == -2) return PKV_ERR_INVALID_ARG;  // groups overlap
    int64_t sp = kv_indptr[first + 1] - kv_indptr[first];
    for (int32_t r = first + 1; r < first + count; ++r) {
      const int64_t n = std::min<int64_t>(sp, kv_indptr[r + 1] - kv_indptr[r]);
      int64_t k = 0;
      while (k < n && kv_indices[kv_indptr[r] + k] == kv_indices[kv_indptr[first] + k]) ++k;
      sp = k;
    }
    for (int32_t r = first; r < first + count; ++r)
      sp = kv_lens[r] < 1 ? 0 : std::min<int64_t>(sp, (kv_lens[r] - 1) / ps);
    if (shared_tokens) shared_tokens[g] = (int32_t)(sp * ps);
    // mark the members (-2: in a group that shares nothing, still counted for overlaps)
    for (int32_t r = first; r < first + count; ++r) owner[r] = sp > 0 ? (int32_t)kept.size() : -2;
    if (sp > 0) kept.push_back({first, count, (int32_t)sp});
  }
  for (int32_t r = 0; r < B; ++r)
    if (owner[r] == -2) owner[r] = -1;

  // splits: as many as one wave of CTAs holds, no chunk shorter than min_chunk_tokens
  int64_t ctas_per_split = 0, max_sp = 0;
  for (const KeptGroup& k : kept) {
    ctas_per_split += (int64_t)num_kv_heads * ((k.count + tpt - 1) / tpt);
    max_sp = std::max<int64_t>(max_sp, k.shared_pages);
  }
  int64_t S = 1;
  if (!kept.empty()) {
    S = std::max<int64_t>(1, ((int64_t)num_sms * ctas_per_sm) / std::max<int64_t>(1, ctas_per_split));
    S = std::max<int64_t>(1, std::min<int64_t>(S, (max_sp * ps) / std::max(1, min_chunk_tokens)));
  }
  if (S * B > INT32_MAX) return PKV_ERR_UNSUPPORTED;

  // count the parts and indices first: a call with no output arrays is a size query
  int64_t nparts = 0, npidx = 0, max_rows = 0;
  for (int32_t r = 0; r < B;) {
    if (owner[r] >= 0) {
      const KeptGroup& k = kept[owner[r]];
      nparts += S;
      npidx += k.shared_pages;
      max_rows = std::max<int64_t>(max_rows, k.count);
      r = k.first + k.count;
    } else {
      int32_t r1 = r;
      while (r1 < B && owner[r1] < 0) ++r1;
      nparts += S;
      max_rows = std::max<int64_t>(max_rows, r1 - r);
      r = r1;
    }
  }
  int64_t nsidx = 0;
  for (int32_t r = 0; r < B; ++r)
    nsidx += (kv_indptr[r + 1] - kv_indptr[r]) - (owner[r] >= 0 ? kept[owner[r]].shared_pages : 0);
  sizes->num_splits = (int32_t)S;
  sizes->num_parts = (int32_t)nparts;
  sizes->max_part_rows = (int32_t)max_rows;
  sizes->num_part_indices = (int32_t)npidx;
  sizes->num_suffix_indices = (int32_t)nsidx;

  int32_t* outs[] = {part_q_start, part_q_len,       part_o_start,     part_kv_indptr, part_kv_indices,
                     part_kv_lens, suffix_kv_indptr, suffix_kv_indices, suffix_kv_lens};
  bool any = false, all = true;
  for (int32_t* p : outs) {
    any = any || p;
    all = all && p;
  }
  if (!any) return PKV_OK;  // size query
  if (!all) return PKV_ERR_INVALID_ARG;
  if (parts_capacity < nparts || indices_capacity < std::max(npidx, nsidx)) return PKV_ERR_WORKSPACE;

  int32_t np = 0, ni = 0;
  part_kv_indptr[0] = 0;
  auto add_part = [&](int32_t r0, int32_t n, int32_t s, const int32_t* pages, int32_t npages) {
    part_q_start[np] = r0;
    part_q_len[np] = n;
    part_o_start[np] = s * B + r0;
    for (int32_t i = 0; i < npages; ++i) part_kv_indices[ni++] = pages[i];
    part_kv_lens[np] = (int32_t)(npages * ps);
    part_kv_indptr[++np] = ni;
  };
  for (int32_t r = 0; r < B;) {
    if (owner[r] >= 0) {
      const KeptGroup& k = kept[owner[r]];
      const int32_t* shared = kv_indices + kv_indptr[k.first];
      const int32_t c = (int32_t)((k.shared_pages + S - 1) / S);  // pages per chunk
      for (int32_t s = 0; s < S; ++s) {
        const int32_t lo = std::min(s * c, k.shared_pages), hi = std::min((s + 1) * c, k.shared_pages);
        add_part(k.first, k.count, s, shared + lo, hi - lo);
      }
      r = k.first + k.count;
    } else {  // rows that share nothing: empty states
      int32_t r1 = r;
      while (r1 < B && owner[r1] < 0) ++r1;
      for (int32_t s = 0; s < S; ++s) add_part(r, r1 - r, s, nullptr, 0);
      r = r1;
    }
  }
  int32_t si = 0;
  suffix_kv_indptr[0] = 0;
  for (int32_t r = 0; r < B; ++r) {
    const int32_t skip = owner[r] >= 0 ? kept[owner[r]].shared_pages : 0;
    for (int32_t k = kv_indptr[r] + skip; k < kv_indptr[r + 1]; ++k) suffix_kv_indices[si++] = kv_indices[k];
    suffix_kv_indptr[r + 1] = si;
    suffix_kv_lens[r] = (int32_t)(kv_lens[r] - skip * ps);
  }
  return PKV_OK;
}
