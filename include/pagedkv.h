/*
 * pagedkv.h -- C ABI of a GB300 (sm_103a) library for attention over a paged KV pool.
 *
 * The operations are the attention layer of an SGLang-style serving engine:
 *   - the paged pool with its page table and token slots (mini-sglang from Scratch handbook,
 *     "What you will be able to do": paged KV pool, page table, token pool);
 *   - K/V of the step's new tokens written into the pool through a slot mapping
 *     (same handbook, "How this book works": the KV-cache writes);
 *   - attention that reads each request's KV in place through page indices, page size 1 or
 *     larger (nanoSGLang README, "Ablation": FlashInfer paged attention, zero-copy KV;
 *     mini-sglang README, "KVcache Management": page size == 1 and > 1);
 *   - GQA and causal attention offset by the cached prefix (Mini-SGLang README,
 *     "Reference Attention Backends", torch backend), with radix-cache prefix pages shared
 *     between requests (mini-sglang README, "KVcache Management": Radix Attention);
 *   - split-KV partial states and their log-sum-exp merge for long decodes.
 *
 * Data layout (all device memory, caller-owned):
 *   pool K and V  bf16 [num_pages, page_size, num_kv_heads, head_dim], contiguous (NHD pages,
 *                 nanoSGLang README, "Architecture").  Flat slot s = page * page_size + row.
 *   page lists    CSR: request b owns pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]), in
 *                 position order; KV position j of request b is row j % page_size of page
 *                 kv_indices[kv_indptr[b] + j / page_size].  Pages may appear in several
 *                 requests' lists (shared prefixes).
 *   GQA           query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   LSE           natural log of sum_j exp(sm_scale * q . k_j), fp32.
 *
 * Calls are asynchronous on the given stream (a cudaStream_t passed as void*, NULL = legacy
 * default stream), never synchronise the host and never allocate: every scratch buffer
 * ("workspace") is passed in by the caller, so a call can be captured in a CUDA graph.  The one
 * exception is pkv_paged_decode_noalloc, which keeps its scratch in an array the library holds on
 * each device; its own comment gives the rules for that array (shared by all its calls, first
 * call on a device before any stream capture).
 *
 * Errors: arguments that can be checked on the host (null pointers, shapes, alignment,
 * workspace size) return a status and launch nothing.  Kernels bounds-check every page index
 * and slot they dereference and skip an access that would fall outside the pool; when
 * err_word is non-NULL they atomically OR a PKV_DEVERR_* bit into that device word.  Waits
 * inside kernels are bounded and report PKV_DEVERR_TIMEOUT instead of hanging.  The caller
 * reads err_word when it chooses to (it is never read by the library).
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, negative count, bad shape or misaligned buffer */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, group size or page size */
  PKV_ERR_WORKSPACE = 3,   /* workspace smaller than the matching *_workspace_size() */
  PKV_ERR_CUDA = 4         /* a CUDA runtime call failed (launch error, no device) */
} pkv_status;

/* Bits OR-ed into *err_word by kernels. */
#define PKV_DEVERR_PAGE_OOB 0x1u /* a page index outside [0, num_pages) was skipped */
#define PKV_DEVERR_SLOT_OOB 0x2u /* an append slot >= num_pages * page_size was skipped */
#define PKV_DEVERR_LENGTH 0x4u   /* a KV length exceeds the request's pages, a decode length is 0,
                                    or an extend / shared-prefix part has more query rows than
                                    max_extend_len / max_part_rows covers (or a negative count) */
#define PKV_DEVERR_TIMEOUT 0x8u  /* a bounded in-kernel wait gave up */
#define PKV_DEVERR_INTERNAL 0x10u /* a launch-time invariant failed and the CTA skipped its work */
#define PKV_DEVERR_ROW_OOB 0x20u   /* a query or output row range outside q / out was skipped */

typedef struct {
  void* k;              /* bf16 [num_pages, page_size, num_kv_heads, head_dim], 16-byte aligned */
  void* v;              /* same shape as k */
  int64_t num_pages;
  int32_t page_size;    /* >= 1 */
  int32_t num_kv_heads; /* >= 1 */
  int32_t head_dim;     /* attention calls: 64 or 128; append/gather: any multiple of 8 */
} pkv_pool;

/* Human-readable name of a status. */
const char* pkv_status_string(pkv_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t pkv_version(void);

/*
 * Host-side checks of step metadata, on HOST copies, before they go to the device: what the
 * kernels would otherwise only report through the error word (or, for duplicate slots, not at
 * all).  Both return PKV_OK, or PKV_ERR_INVALID_ARG with the first offending request / token in
 * *bad_request / *bad_token (nullable; -1 when none).
 *
 * pkv_validate_page_table: kv_indptr[0] == 0 and non-decreasing; every listed page index in
 * [0, num_pages); min_len <= kv_lens[b] <= (kv_indptr[b+1] - kv_indptr[b]) * page_size (min_len
 * 1 for a decode; for an extend pass the KV lengths prefix + new tokens and min_len 1).
 *   kv_indptr int32 [batch_size+1], kv_indices int32 [kv_indptr[batch_size]], kv_lens int32
 *   [batch_size] (host)
 *
 * pkv_validate_slots: every slot < num_slots (= num_pages * page_size); negative slots are
 * padding; no slot written twice (the append's caller contract).  *bad_token is the first
 * out-of-range token, else the first token whose slot an earlier token already writes.
 *   slot_mapping int64 [num_tokens] (host)
 */
pkv_status pkv_validate_page_table(const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* kv_lens, int32_t batch_size, int64_t num_pages,
                                   int32_t page_size, int32_t min_len, int32_t* bad_request);
pkv_status pkv_validate_slots(const int64_t* slot_mapping, int32_t num_tokens, int64_t num_slots,
                              int32_t* bad_token);

/*
 * Check of the kernels' failure path: one GPU thread waits on an mbarrier that nothing ever
 * arrives on, with the bounded wait every kernel of this library uses (0.5 s of %globaltimer),
 * then gives up and ORs PKV_DEVERR_TIMEOUT into *err_word (device uint32, required).  The launch
 * returns at once; after the stream synchronises the word holds the bit and the context stays
 * usable.  It exists so that tests can show that a wait that never completes ends with an error
 * status instead of a hang.
 */
pkv_status pkv_selftest_bounded_wait(uint32_t* err_word, void* stream);

/*
 * KV-cache write.  For t < num_tokens: pool.k row slot_mapping[t] = k_new[t] and the same for
 * V; a negative slot marks a padding token and writes nothing.  A bit-exact copy.
 *   k_new, v_new  bf16 [num_tokens, num_kv_heads, head_dim] (device)
 *   slot_mapping  int64 [num_tokens] (device); slots must be distinct within one call
 *   err_word      nullable device uint32; PKV_DEVERR_SLOT_OOB for slot >= num_pages*page_size
 */
pkv_status pkv_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int32_t num_tokens, uint32_t* err_word,
                         void* stream);

/*
 * KV-cache write fused with the rotary position embedding of the step's new tokens (the step
 * just before attention in the engines' forward pass).  For t < num_tokens, with p = positions[t]:
 *   pool.k row slot_mapping[t] = bf16(rope(k_new[t], p)),  pool.v row slot_mapping[t] = v_new[t],
 *   and, when q is not NULL, q[t] = bf16(rope(q[t], p)) in place.
 * rope is the half-split pairing of HF Llama/Qwen checkpoints (nanoSGLang README, "Notable
 * Fixes"): for i < head_dim/2, x'[i] = x[i] cos a_i - x[i+D/2] sin a_i and
 * x'[i+D/2] = x[i+D/2] cos a_i + x[i] sin a_i, computed in fp32 and rounded to nearest even.
 *   cos_sin       fp32 [max_position, head_dim] (device): row p holds cos(a_i) in columns
 *                 [0, D/2) and sin(a_i) in [D/2, D), a_i = p * theta^(-2i/D); built once by the caller
 *   positions     int32 [num_tokens] (device); a position outside [0, max_position) skips that
 *                 token's writes and reports PKV_DEVERR_LENGTH
 *   q             nullable bf16 [num_tokens, num_q_heads, head_dim], rotated in place
 *   slot_mapping, k_new, v_new, err_word as for pkv_kv_append.  head_dim a multiple of 16.
 */
pkv_status pkv_rope_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, const int32_t* positions,
                              const float* cos_sin, int32_t max_position, void* q,
                              int32_t num_q_heads, int32_t num_tokens, uint32_t* err_word,
                              void* stream);

/*
 * The cos/sin table pkv_rope_kv_append reads, computed on the device.  Row p of
 * table fp32 [max_position, head_dim] (device, caller-owned) receives cos(a_i) in columns
 * [0, D/2) and sin(a_i) in [D/2, D), a_i = p * theta^(-2i/D) (the half-split rotary embedding of
 * HF Llama/Qwen checkpoints, nanoSGLang README "Notable Fixes").  The angle is formed in double
 * precision and cos/sin are rounded once to fp32.  head_dim even, theta > 0 (e.g. 1e4 for
 * Llama, 1e6 for Qwen3), max_position >= 0 (0 launches nothing).  Asynchronous on the stream.
 */
pkv_status pkv_rope_cos_sin_table(float* table, int32_t max_position, int32_t head_dim, double theta,
                                  void* stream);

/*
 * Page gather (test and debug op): copy every request's K and V rows, in position order, into
 * contiguous buffers.  Request b occupies rows [sum_{b'<b} kv_lens[b'], ... + kv_lens[b]).
 *   kv_indptr  int32 [batch_size+1], kv_indices int32 [kv_indptr[batch_size]], kv_lens int32
 *              [batch_size] (device)
 *   k_out, v_out  bf16 [sum(kv_lens), num_kv_heads, head_dim] (device)
 *   err_word   nullable; PKV_DEVERR_PAGE_OOB / PKV_DEVERR_LENGTH, the row is left unwritten
 */
pkv_status pkv_paged_gather(const pkv_pool* pool, const int32_t* kv_indptr,
                            const int32_t* kv_indices, const int32_t* kv_lens, int32_t batch_size,
                            void* k_out, void* v_out, uint32_t* err_word, void* stream);

/*
 * Bytes of workspace pkv_paged_decode needs for this shape on the current device (the split
 * partials, sized by the device's SM count).  Returns 0 for an invalid shape.
 */
size_t pkv_decode_workspace_size(int32_t batch_size, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim);

/*
 * Paged decode: one query per request at its last position, attending over all kv_lens[b]
 * positions (the KV of the step's own token is appended first with pkv_kv_append).
 *   q          bf16 [batch_size, num_q_heads, head_dim] (device)
 *   kv_indptr, kv_indices, kv_lens  as for pkv_paged_gather; kv_lens[b] >= 1
 *   sm_scale   softmax scale applied to q . k (e.g. 1/sqrt(head_dim))
 *   out        bf16 [batch_size, num_q_heads, head_dim] (device), round-to-nearest-even
 *   lse        nullable fp32 [batch_size, num_q_heads] (device)
 *   workspace  device buffer of at least pkv_decode_workspace_size(...) bytes, 256-byte
 *              aligned; its contents need no initialisation and are clobbered
 * Long requests are split across CTAs (flash-decoding) and merged by log-sum-exp in a second
 * kernel on the same stream.  head_dim 64 or 128, num_q_heads / num_kv_heads <= 16.
 * A request with kv_lens[b] == 0 gets out = 0, lse = -inf and PKV_DEVERR_LENGTH.
 */
pkv_status pkv_paged_decode(const pkv_pool* pool, const void* q, int32_t batch_size,
                            int32_t num_q_heads, const int32_t* kv_indptr,
                            const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            uint32_t* err_word, void* stream);

/*
 * pkv_paged_decode on at most max_ctas SMs: one persistent CTA per SM as always, but only
 * max_ctas of them (0, or a value at or above the SM count, means every SM; negative is
 * PKV_ERR_INVALID_ARG).  The other SMs stay free for kernels on other streams.  The decode is
 * bound by HBM bandwidth, which a few SMs fewer still nearly saturate, so a tensor-core kernel
 * running beside it (the step's extend, on its own stream) gains those SMs for little decode
 * time.  Same arguments, workspace size, results and errors as pkv_paged_decode, whose call is
 * this one with max_ctas = 0.
 */
pkv_status pkv_paged_decode_ctas(const pkv_pool* pool, const void* q, int32_t batch_size,
                                 int32_t num_q_heads, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 uint32_t* err_word, int32_t max_ctas, void* stream);

/*
 * pkv_paged_decode_ctas with an L2 residency hint for KV that several requests of the batch read:
 * the pages of a prefix shared through the radix cache (mini-sglang README, "KVcache
 * Management").  The decode streams every request's KV through L2 once; without a hint, a shared
 * prefix read early in the step is evicted by the stream before the sharers that come later read
 * it, and it is fetched from HBM again for them.
 *   keep_tokens  nullable device int32 [batch_size]: request b's positions below keep_tokens[b]
 *                are fetched with an evict-last L2 policy (the caller expects other requests of
 *                the batch to read them too, e.g. its radix-cache match length when the match is
 *                shared), every other position with evict-first.  NULL: the default policy for
 *                every load, which is pkv_paged_decode_ctas.
 * The hint only steers what the L2 evicts: results are bit for bit those of pkv_paged_decode_ctas
 * with the same arguments, whatever keep_tokens holds.  Marking unshared KV evict-last makes it
 * crowd the shared pages out instead, and marking a shared prefix 0 makes it leave first.
 */
pkv_status pkv_paged_decode_l2keep(const pkv_pool* pool, const void* q, int32_t batch_size,
                                   int32_t num_q_heads, const int32_t* kv_indptr,
                                   const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                                   uint32_t* err_word, int32_t max_ctas, const int32_t* keep_tokens,
                                   void* stream);

/*
 * Decode for callers that cannot allocate device memory.  No counterpart on the pages: this is a
 * convenience of this library.  A serving engine that reserves a fixed share of HBM for its KV
 * pool, or code that must not call cudaMalloc (and take its implicit device synchronisation) in
 * the middle of a step, has no workspace to pass to pkv_paged_decode.  This entry point takes the
 * same arguments minus the workspace and uses a scratch array that the library holds in device
 * memory: PKV_DECODE_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, until the
 * process exits.  It allocates nothing itself.
 *   - Shapes whose pkv_decode_workspace_size() exceeds PKV_DECODE_NOALLOC_SCRATCH_BYTES are
 *     rejected with PKV_ERR_WORKSPACE (Hq=32, head_dim 128 fits about 800 requests).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, which
 *     may load the module on that device); make that first call before any stream capture.  A
 *     device reset (cudaDeviceReset) frees the array with its context: the next call on that
 *     device looks the address up again and, like a first call, must come before any capture.
 *   - Every call shares the one array and it keeps the last call's contents; nothing in it needs
 *     to start at zero.  Calls that can overlap on the GPU (different streams without ordering)
 *     race on it: serialise them.
 * Results are those of pkv_paged_decode with the same arguments.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
pkv_status pkv_paged_decode_noalloc(const pkv_pool* pool, const void* q, int32_t batch_size,
                                    int32_t num_q_heads, const int32_t* kv_indptr,
                                    const int32_t* kv_indices, const int32_t* kv_lens,
                                    float sm_scale, void* out, float* lse, uint32_t* err_word,
                                    void* stream);

/*
 * Bytes of workspace pkv_paged_extend needs: the order in which its grid visits the requests
 * (longest KV first), int32 per request, for batches of 33 to 4096 requests.  0 for up to 32
 * requests (the kernel ranks them itself) and above 4096 (batch order).
 */
size_t pkv_extend_workspace_size(int32_t batch_size, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_extend_len);

/*
 * Ragged extend (prefill / chunked prefill over a cached prefix).  Request b's queries are rows
 * qo_indptr[b] .. qo_indptr[b+1] of q; query i of the request is at absolute position
 * prefix_lens[b] + i and attends to KV positions j <= prefix_lens[b] + i.  The request's KV
 * length is prefix_lens[b] + (qo_indptr[b+1] - qo_indptr[b]) and all of it is read through the
 * pool: append the new tokens' K/V first.
 *   q          bf16 [num_q_tokens, num_q_heads, head_dim] (device)
 *   num_q_tokens  rows of q and out (= qo_indptr[batch_size])
 *   qo_indptr  int32 [batch_size+1]; prefix_lens int32 [batch_size] (device)
 *   max_extend_len  an upper bound of qo_indptr[b+1]-qo_indptr[b] over b (sizes the grid).
 *              A request with more rows than the grid covers, or with qo_indptr decreasing,
 *              reports PKV_DEVERR_LENGTH and its rows past the grid are left unwritten.
 *   out        bf16 [num_q_tokens, num_q_heads, head_dim]; lse nullable fp32 [num_q_tokens, num_q_heads]
 *   workspace  device, 16-byte aligned, at least pkv_extend_workspace_size(...) bytes, caller-owned
 *              and not shared with a call in flight on another stream (may be NULL when that
 *              size is 0); smaller returns PKV_ERR_WORKSPACE
 * head_dim 64 or 128, any page_size (powers of two >= 8 are gathered by TMA boxes, others row by
 * row), num_q_heads / num_kv_heads from 1 to 16 (a Q tile holds group x floor(128 / group) rows of
 * (token, query head) pairs).
 */
pkv_status pkv_paged_extend(const pkv_pool* pool, const void* q, int32_t num_q_tokens,
                            const int32_t* qo_indptr, int32_t batch_size, int32_t num_q_heads,
                            const int32_t* kv_indptr, const int32_t* kv_indices,
                            const int32_t* prefix_lens, int32_t max_extend_len, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            uint32_t* err_word, void* stream);

/*
 * Bytes of workspace pkv_shared_prefix_attention needs (the order of its parts, as for the extend).
 */
size_t pkv_shared_prefix_workspace_size(int32_t num_parts, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t max_part_rows);

/*
 * Shared-prefix (cascade) attention.  When several requests share the first pages of their KV
 * (radix-cache prefix sharing: mini-sglang README, "KVcache Management"), the attention of all
 * their queries over those pages is computed together, so each shared page is read once per
 * part instead of once per request, and on tensor cores.  The result is a partial state of each
 * query over the shared positions, merged with the partial state over the request's own pages
 * (a decode over the suffix page list) by pkv_merge_states_bf16; split the shared pages over
 * several parts to spread long prefixes over the GPU.
 * Part p: query rows q_start[p] .. q_start[p] + q_len[p] - 1 of q attend, without a mask, to all
 * kv_lens[p] positions of page list p (kv_indptr / kv_indices as for the decode), with GQA as in
 * the extend; the part's output rows are o_start[p] .. o_start[p] + q_len[p] - 1 of o_part:
 *   o_part[r, h, :] = sum_j softmax_j(scale * q . k_j) v_j,  lse_part[r, h] = ln sum_j exp(scale * q . k_j)
 * A part with kv_lens[p] == 0 writes o = 0 and lse = -inf (an empty split for the merge).
 *   q          bf16 [num_q_rows, num_q_heads, head_dim] (device)
 *   q_start, q_len, o_start, kv_lens  int32 [num_parts]; kv_indptr int32 [num_parts+1] (device)
 *   max_part_rows  an upper bound of q_len[p] (sizes the grid); a longer or negative part reports
 *              PKV_DEVERR_LENGTH and its rows past the grid are left unwritten
 *   o_part     bf16 [num_out_rows, num_q_heads, head_dim]; lse_part nullable fp32 [num_out_rows, num_q_heads]
 *   workspace  as for pkv_paged_extend, pkv_shared_prefix_workspace_size(...) bytes
 *   err_word   nullable; PKV_DEVERR_ROW_OOB for a part whose rows fall outside q or o_part (the part
 *              is skipped), PKV_DEVERR_PAGE_OOB / PKV_DEVERR_LENGTH as for the extend
 * head_dim 64 or 128, any page_size, group size 1 to 16.  Parts that write
 * the same output rows race; different parts may read the same query rows.
 */
pkv_status pkv_shared_prefix_attention(const pkv_pool* pool, const void* q, int32_t num_q_rows,
                                       const int32_t* q_start, const int32_t* q_len,
                                       const int32_t* o_start, int32_t num_parts, int32_t num_q_heads,
                                       const int32_t* kv_indptr, const int32_t* kv_indices,
                                       const int32_t* kv_lens, int32_t max_part_rows, float sm_scale,
                                       void* o_part, float* lse_part, int32_t num_out_rows,
                                       void* workspace, size_t workspace_bytes, uint32_t* err_word,
                                       void* stream);

/*
 * Host plan of a shared-prefix (cascade) decode: the integer arrays pkv_shared_prefix_attention,
 * pkv_paged_decode and pkv_merge_states_bf16 take, computed on the CPU from HOST copies of the
 * decode batch's page lists (the "plan" of a plan/run split: mini-sglang from Scratch handbook,
 * "What you will be able to do").  No attention arithmetic happens here.
 *
 * Groups g < num_groups are runs of consecutive requests [group_first[g], + group_count[g]) that
 * share leading pages (radix-cache prefixes).  A group's shared length is the longest common
 * leading run of page ids of its members, cut so that every member keeps at least one position
 * of its own; shared_tokens[g] (nullable, [num_groups]) receives it in positions, 0 for a group
 * that shares nothing (then treated as unshared).  The shared pages of every group are cut into
 * the same number S of chunks (sizes->num_splits): as many as one wave of CTAs covers
 * (num_sms * ctas_per_sm over num_kv_heads * ceil(members / (128 / group_size)) CTAs per chunk),
 * and no chunk shorter than min_chunk_tokens.
 *
 * Partial states are laid out as splits of one buffer [S + 1, batch_size, Hq, ...]: split s < S
 * of row r is chunk s of r's group (an empty state for rows outside every group and chunks a
 * group does not have), split S is the decode over r's own pages.
 *   part p (p < num_parts):  query rows part_q_start[p] .. + part_q_len[p]; output rows
 *     part_o_start[p] = s * batch_size + part_q_start[p]; page list part_kv_indices
 *     [part_kv_indptr[p] .. part_kv_indptr[p+1]) with part_kv_lens[p] = its pages * page_size
 *     (0 for an empty state)
 *   own pages of request r:  suffix_kv_indices[suffix_kv_indptr[r] .. suffix_kv_indptr[r+1]),
 *     suffix_kv_lens[r] >= 1 positions
 * Inputs (host): kv_indptr int32 [batch_size+1] (kv_indptr[0] == 0, non-decreasing), kv_indices
 * int32 [kv_indptr[batch_size]], kv_lens int32 [batch_size].  group_size = Hq / Hkv in 1..16.
 * Outputs (host, caller-owned): sizes (required) receives the counts.  With every output array
 * NULL the call only fills sizes (a size query).  Otherwise all nine arrays are required:
 * part_* of parts_capacity entries (part_kv_indptr one more), part_kv_indices and
 * suffix_kv_indices of indices_capacity entries (kv_indptr[batch_size] always suffices),
 * suffix_kv_indptr [batch_size+1], suffix_kv_lens [batch_size]; too small a capacity returns
 * PKV_ERR_WORKSPACE with sizes filled.  Groups outside the batch or overlapping, and bad counts,
 * return PKV_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t num_splits;         /* S: shared-prefix chunks; the own-pages decode is split S */
  int32_t num_parts;          /* parts of pkv_shared_prefix_attention */
  int32_t max_part_rows;      /* the largest part_q_len (its max_part_rows argument) */
  int32_t num_part_indices;   /* entries written to part_kv_indices */
  int32_t num_suffix_indices; /* entries written to suffix_kv_indices */
} pkv_cascade_sizes;

pkv_status pkv_plan_shared_prefix(const int32_t* kv_indptr, const int32_t* kv_indices,
                                  const int32_t* kv_lens, int32_t batch_size,
                                  const int32_t* group_first, const int32_t* group_count,
                                  int32_t num_groups, int32_t page_size, int32_t num_kv_heads,
                                  int32_t group_size, int32_t num_sms, int32_t ctas_per_sm,
                                  int32_t min_chunk_tokens, pkv_cascade_sizes* sizes,
                                  int32_t* shared_tokens, int32_t* part_q_start, int32_t* part_q_len,
                                  int32_t* part_o_start, int32_t* part_kv_indptr,
                                  int32_t* part_kv_indices, int32_t* part_kv_lens,
                                  int32_t* suffix_kv_indptr, int32_t* suffix_kv_indices,
                                  int32_t* suffix_kv_lens, int32_t parts_capacity,
                                  int32_t indices_capacity);

/*
 * Log-sum-exp merge of split partial states (flash-decoding).  For each row n and head h:
 *   lse[n,h] = ln sum_s exp(lse_parts[s,n,h]);  out[n,h,:] = sum_s exp(lse_parts[s,n,h] - lse[n,h]) * o_parts[s,n,h,:]
 * A split with lse_parts = -inf is empty and contributes nothing; if all are empty the row gets
 * out = 0, lse = -inf.
 *   o_parts    fp32 [num_splits, num_rows, num_heads, head_dim] (device), each split normalised
 *              by its own softmax sum
 *   lse_parts  fp32 [num_splits, num_rows, num_heads] (device)
 *   out        bf16 [num_rows, num_heads, head_dim]; lse nullable fp32 [num_rows, num_heads]
 * head_dim a multiple of 4, at most 512.
 */
pkv_status pkv_merge_states(const float* o_parts, const float* lse_parts, int32_t num_splits,
                            int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                            float* lse, void* stream);

/*
 * pkv_merge_states with bf16 partial outputs, o_parts bf16 [num_splits, num_rows, num_heads,
 * head_dim] (16-byte aligned), e.g. the shared-prefix parts and a decode over each request's own
 * pages written into consecutive splits.  Accumulates in fp32.
 */
pkv_status pkv_merge_states_bf16(const void* o_parts, const float* lse_parts, int32_t num_splits,
                                 int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                                 float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
