// Ragged extend attention (prefill / chunked prefill over a cached prefix) on tcgen05 tensor cores.
//
// What it computes: request b's E_b new tokens attend causally to its KV, read in place from the
// paged pool; query i sits at absolute position P_b + i and sees positions j <= P_b + i (the
// causal mask offset by the cached prefix, Mini-SGLang README "Reference Attention Backends",
// torch backend), with GQA (query head h reads KV head h / G) and prefix pages that several
// requests share (mini-sglang README, "KVcache Management": Radix Attention).  Chunked prefill
// (nanoLLMServe README, "v0.7 Chunked Prefill") is the same call with a non-zero prefix.
//
// Design for GB300:
//  * One CTA per (128-row Q tile, KV head, request).  The rows are (token, group head) pairs:
//    floor(128/G) consecutive tokens times the G query heads that share the KV head (G from 1
//    to 16), so each K/V tile loaded is used by the whole group.  Q arrives by one 3-D TMA box
//    per 64-column half (head_dim 64 or 128).  A batch of up to 32 requests is ranked (longest KV
//    first) inside the kernel and takes a compact grid, one CTA per Q tile it has, the kv heads of
//    a tile dispatched together; larger batches take a grid sized by max_extend_len.
//  * K and V tiles of 64 positions are gathered page by page with 3-D TMA boxes
//    [64 dims x 1 head x min(page,64) rows] in 128-byte swizzle (other page sizes: row copies
//    into the same layout), into 2-stage rings filled by two producer warps (K with Q, and V), so
//    the K stream runs ahead of the V stream.
//  * S = Q K^T (M=128, N=64, K=128) and O += P V (M=128, N=128, K=64) run as tcgen05.mma,
//    accumulating in TMEM: S double-buffered (2 x 64 columns), O in 128 columns.  QK and PV are
//    issued by two threads in different warps, each blocked in a try_wait on its own operands, so
//    a PV whose P is ready starts within a few hundred cycles instead of waiting behind a QK.
//    A tcgen05.mma issue costs about as long as an N=128 MMA whatever its N, so PV is issued as
//    one N=128 MMA per 16 positions rather than two of N=64.
//    P is written back as bf16 pairs over the S columns it came from and the PV MMA reads it from
//    TMEM, so P never passes through shared memory.
//  * Four softmax warps, one per TMEM lane quadrant: a thread owns one row of the tile and reads
//    all 64 of its scores, so the row max needs no exchange between warps (a three-input max.f32
//    folds three scores per instruction).  It applies the causal mask and the online softmax in
//    fp32 (the running max only moves when it grows by more than 2^8, so O is rescaled in TMEM
//    rarely), keeps two sums of the probabilities (the exact one for the LSE; the one of the bf16
//    values the PV MMA uses, accumulated straight from the packed bf16 pairs by the sm_100
//    family's mixed-precision add, for O).  At the end all eight warps normalise the O tile into
//    shared memory in the Q box layout, half a row each, and it leaves by TMA tensor stores (a
//    request's last, partial tile by coalesced stores of all threads).
//  * Two CTAs fit on an SM (99 KB of shared memory and 256 TMEM columns each), so one CTA's
//    softmax overlaps the other's MMAs.
#include <algorithm>
#include <atomic>

#include "tc05.cuh"

namespace {

using namespace pkv;

constexpr int kBM = 128;  // Q tile rows: (token, group head) pairs
constexpr int kBN = 64;   // KV positions per tile
// warp 0 Q/K loads, warp 1 QK MMAs, warps 2..5 softmax (one per TMEM lane quadrant, a thread
// per row of the tile), warp 6 V loads, warp 7 PV MMAs
constexpr int kSoftmaxWarps = 4;
constexpr int kVWarp = 2 + kSoftmaxWarps;
constexpr int kPVWarp = kVWarp + 1;
constexpr int kThreads = (kPVWarp + 1) * 32;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;  // O at TMEM columns [128, 128 + D); S buffers at [0,64) and [64,128)
constexpr uint32_t kQHalf = kBM * 128;   // one 64-dim half of the Q tile, 16 KB
constexpr uint32_t kKVHalf = kBN * 128;  // 64 positions x 64 dims, 8 KB

// Shared-memory layout for head_dim D (64 or 128): operands are stored as 64-dim halves of
// 128-byte swizzled rows.
template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQBytes = kHalves * kQHalf;  // also the O staging tile (128 rows x 2D bytes)
  static constexpr uint32_t kKVStage = kHalves * kKVHalf;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffK + 2 * kKVStage;
  static constexpr uint32_t kOffBar = kOffV + 2 * kKVStage;
  static constexpr uint32_t kOffInv = kOffBar + 256;  // 1 / (sum of P) of each tile row, fp32
  static constexpr uint32_t kSmemBytes = kOffInv + kBM * 4;
  static constexpr int kChunks = D * 2 / 16;  // 16-byte chunks of an O row
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2];  // S buffer b: QK written / its P consumed by PV
  uint64_t p_full[2];              // P of the tile in S buffer b written by the softmax
  uint64_t qk_done, pv_done;       // every MMA of the issuing thread has completed (exit path)
  uint32_t tmem_base;
  uint32_t epi_skip;  // set by a softmax thread whose waits gave up: no O to write
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct ExtendArgs {
  CUtensorMap tm_q;
  CUtensorMap tm_o;  // out viewed like q: the box of a full Q tile is stored by TMA
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* prefix_lens;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* err_word;
  int64_t num_pages;
  int32_t page_size;
  int32_t log2_ps;
  int32_t num_q_heads;
  int32_t group;
  int32_t rows_used;   // group * tokens_per_tile <= 128 Q-tile rows hold (token, head) pairs
  int32_t log2_group;  // log2(group) when the group is a power of two, else -1 (divide)
  int32_t tokens_per_tile;
  float scale_log2;
  const int32_t* order;  // request of grid z-index z, longest KV first (nullable: ranked in the
                         // kernel when rank_inline, else batch order)
  int32_t rank_inline;   // batch_size <= 32: each warp ranks the requests itself
  int32_t compact;       // (causal, ranked in the kernel) grid (kv heads, Q tiles of all requests)
  int32_t max_tiles;     // Q tiles per request the call covers: ceil(max_extend_len / tokens_per_tile)
  int32_t batch;         // requests (or parts)
  // shared-prefix parts (the unmasked instance): part b's rows q_start[b] .. + q_len[b] of q attend to all
  // prefix_lens[b] positions of its page list and write rows o_start[b] .. of out
  const int32_t* q_start;
  const int32_t* o_start;
  const int32_t* q_len;
  int32_t num_q_rows;    // rows of q
  int32_t num_out_rows;  // rows of out
  // the pool, for the row-copy producer (page sizes that are not a power of two >= 8)
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int32_t num_kv_heads;
};

struct Work {
  // q0 / qo0: first query row of the request in q / in out; row i of the request sees the KV
  // positions j <= min(mask0 + i, L - 1); p0 / np: its page list's offset and length
  int h, b, q0, qo0, E, P, p0, np, t0, mask0, L, kv_end, n_tiles;
};

// A request's (or part's) metadata: its rows, KV length and page list, as one round of
// independent loads.
template <bool kCausal>
__device__ __forceinline__ void load_request(const ExtendArgs& a, int b, Work& w) {
  if (kCausal) {
    w.qo0 = __ldg(a.qo_indptr + b);
    w.E = __ldg(a.qo_indptr + b + 1) - w.qo0;
    w.q0 = w.qo0;
  } else {
    w.q0 = __ldg(a.q_start + b);
    w.qo0 = __ldg(a.o_start + b);
    w.E = __ldg(a.q_len + b);
  }
  w.P = __ldg(a.prefix_lens + b);
  w.p0 = __ldg(a.kv_indptr + b);
  w.np = __ldg(a.kv_indptr + b + 1) - w.p0;
}

// The request's page list as the TMA producers read it: its offset and length, and a register
// window of 64 entries (lane i holds entries i and 32 + i), loaded before the CTA's set-up
// barrier so that the first K/V boxes do not wait on it.
struct PageWindow {
  int32_t w0, w1;
};

__device__ __forceinline__ PageWindow load_page_window(const ExtendArgs& a, const Work& w) {
  const int lane = threadIdx.x & 31;
  PageWindow pw;
  pw.w0 = lane < w.np ? __ldg(a.kv_indices + w.p0 + lane) : -1;
  pw.w1 = 32 + lane < w.np ? __ldg(a.kv_indices + w.p0 + 32 + lane) : -1;
  return pw;
}

// Producer warp: Q once, then K and V tiles page by page.  Lane i issues box i of a tile; the
// page indices come from a register window of 64 page-list entries whose upper half is loaded
// 32 pages before it is needed, so no TMA waits on a dependent global load.
// kv = 0: the K warp (also loads Q); kv = 1: the V warp.  Separate warps keep the K stream
// ahead of the QK MMAs even while the V stream waits for its stage to be freed by PV.  The
// warp returns only when its copies have landed (bounded waits).
template <int D>
__device__ bool extend_producer(const ExtendArgs& a, uint32_t sb, Bars* bars, const Work& w, int kv,
                                const PageWindow& pw) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int p0 = w.p0, np = w.np;
  const int R = min(a.page_size, kBN);  // rows per box (a power of two, >= 8)
  const int nbox = kBN / R;             // boxes per tile (<= 8)
  auto entry = [&](int pidx) -> int32_t {
    return (pidx >= 0 && pidx < np) ? __ldg(a.kv_indices + p0 + pidx) : -1;
  };
  uint64_t* fulls = kv ? bars->v_full : bars->k_full;
  uint64_t* empties = kv ? bars->v_empty : bars->k_empty;
  const CUtensorMap* tm = kv ? &a.tm_v : &a.tm_k;
  int wbase = 0;
  int32_t w0 = pw.w0, w1 = pw.w1;
  int issued = 0;
  bool ok = true;
  for (int j = 0; j < w.n_tiles; ++j) {
    const int st = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    // box `lane` of tile j: positions [pos0, pos0 + R)
    const int pos0 = j * kBN + lane * R;
    const int pidx = pos0 >> a.log2_ps;
    while ((j * kBN >> a.log2_ps) >= wbase + 32) {
      w0 = w1;
      wbase += 32;
      w1 = entry(wbase + 32 + lane);
    }
    const int k = pidx - wbase;  // < 64: a tile spans at most 8 pages past the window base
    const int32_t v0 = __shfl_sync(0xffffffffu, w0, k & 31);
    const int32_t v1 = __shfl_sync(0xffffffffu, w1, k & 31);
    const int32_t page = k < 32 ? v0 : v1;
    int row = -1;
    if (lane < nbox && pos0 < w.kv_end) {
      if (pidx >= np)
        report(a.err_word, PKV_DEVERR_LENGTH);
      else if (page < 0 || page >= a.num_pages)
        report(a.err_word, PKV_DEVERR_PAGE_OOB);
      else
        row = (int)((int64_t)page * a.page_size + (pos0 & (a.page_size - 1)));
    }
    const uint32_t nload = __popc(__ballot_sync(0xffffffffu, row >= 0));
    if (!__all_sync(0xffffffffu, mbar_wait(&empties[st], ph ^ 1))) {
      if (lane == 0) report(a.err_word, PKV_DEVERR_TIMEOUT);
      ok = false;
      break;
    }
    if (lane == 0) mbar_arrive_expect_tx(&fulls[st], nload * R * 128 * C::kHalves);
    __syncwarp();
    if (row >= 0) {
      const uint32_t dst = sb + (kv ? C::kOffV : C::kOffK) + st * C::kKVStage + lane * R * 128;
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf) tma_load_3d(dst + hf * kKVHalf, tm, hf * 64, w.h, row, &fulls[st]);
    }
    issued = j + 1;
  }
  // no copy of this warp is in flight when the CTA exits, also after a timeout elsewhere
  // (immediate on the normal path, where the MMAs have consumed every tile)
  for (int j = max(0, issued - 2); j < issued; ++j) mbar_wait(&fulls[j & 1], (j >> 1) & 1);
  if (kv == 0) mbar_wait(&bars->q_full, 0);
  return ok;
}

// 16-byte asynchronous copies global -> shared (cache in L2 only), committed and waited per
// group; the producer makes them visible to the tensor cores with a proxy fence.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Producer for any page size (used when it is not a power of two >= 8, page size 1 included): the
// 64 rows of a K or V tile are copied one token row at a time, two rows per lane, 16 bytes per
// cp.async, into the same 128-byte-swizzled layout the TMA boxes produce (chunk c of row r at
// chunk c ^ (r % 8)).  A stage is announced on its full barrier once its copies have landed:
// after issuing stage j the warp waits for stage j-1's group, fences the async proxy (the MMAs
// read shared memory through it) and arrives.  The page indices of the next tile are loaded
// while the current one is copied.  Q still comes by TMA.
template <int D>
__device__ bool extend_producer_rows(const ExtendArgs& a, uint32_t sb, Bars* bars, const Work& w, int kv) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int p0 = w.p0, np = w.np;
  const int ps = a.page_size;
  const __nv_bfloat16* pool = kv ? a.v_pool : a.k_pool;
  uint64_t* fulls = kv ? bars->v_full : bars->k_full;
  uint64_t* empties = kv ? bars->v_empty : bars->k_empty;
  // slot of this lane's row rr of tile j, or -1 (past the KV end, or a bad index, reported)
  auto slot_of = [&](int j, int rr) -> int64_t {
    const int pos = j * kBN + lane + 32 * rr;
    if (j >= w.n_tiles || pos >= w.kv_end) return -1;
    const int pidx = pos / ps;
    if (pidx >= np) {
      report(a.err_word, PKV_DEVERR_LENGTH);
      return -1;
    }
    const int32_t page = __ldg(a.kv_indices + p0 + pidx);
    if (page < 0 || page >= a.num_pages) {
      report(a.err_word, PKV_DEVERR_PAGE_OOB);
      return -1;
    }
    return (int64_t)page * ps + (pos - pidx * ps);
  };
  int64_t s0 = slot_of(0, 0), s1 = slot_of(0, 1);
  int issued = 0;
  bool ok = true;
  for (int j = 0; j < w.n_tiles; ++j) {
    const int st = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    if (!__all_sync(0xffffffffu, mbar_wait(&empties[st], ph ^ 1))) {
      if (lane == 0) report(a.err_word, PKV_DEVERR_TIMEOUT);
      ok = false;
      break;
    }
    const uint32_t base = sb + (kv ? C::kOffV : C::kOffK) + st * C::kKVStage;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int64_t slot = rr ? s1 : s0;
      if (slot >= 0) {
        const int row = lane + 32 * rr;
        const char* src = reinterpret_cast<const char*>(pool + (slot * a.num_kv_heads + w.h) * D);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            cp_async16(base + hf * kKVHalf + row * 128 + ((c ^ (row & 7)) << 4), src + hf * 128 + c * 16);
      }
    }
    cp_async_commit();
    issued = j + 1;
    s0 = slot_of(j + 1, 0);  // the next tile's rows, while these copies fly
    s1 = slot_of(j + 1, 1);
    if (j > 0) {  // the previous stage has landed: publish it
      cp_async_wait_group<1>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&fulls[(j - 1) & 1]);
    }
  }
  // the last stage issued (also after a timeout: no copy of this warp is left in flight)
  cp_async_wait_group<0>();
  fence_proxy_async_smem();
  __syncwarp();
  if (issued > 0 && lane == 0) mbar_arrive(&fulls[(issued - 1) & 1]);
  if (kv == 0) mbar_wait(&bars->q_full, 0);
  return ok;
}

// The MMAs are issued by two threads, one per stream, each waiting with a blocking try_wait that
// wakes when its phase completes:  the QK thread issues QK(j) once K(j) has landed and S buffer
// j&1 is back from PV(j-2) (P is written over S);  the PV thread issues PV(j) once the softmax
// has written P(j) and V(j) has landed.  Neither stream ever waits behind the other.
template <int D>
__device__ bool extend_mma_qk(const ExtendArgs& a, uint32_t sb, Bars* bars, uint32_t tmem, const Work& w) {
  using C = Cfg<D>;
  constexpr uint32_t idesc_qk = umma_idesc_bf16(kBM, kBN, false);
  // operand descriptors built once: a K-step or a stage only moves the start address field
  // (address / 16 in the low 14 bits; every offset here stays inside shared memory's 256 KB)
  const uint64_t qdesc = smem_desc_sw128(sb + C::kOffQ, 16, 1024);
  const uint64_t kdesc0 = smem_desc_sw128(sb + C::kOffK, 16, 1024);
  if (!mbar_wait(&bars->q_full, 0)) return false;
  for (int j = 0; j < w.n_tiles; ++j) {
    const int st = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    if (!mbar_wait(&bars->k_full[st], ph)) return false;
    if (!mbar_wait(&bars->s_free[st], ph ^ 1)) return false;
    tc_fence_after();
    const uint64_t kdesc = kdesc0 + ((st * C::kKVStage) >> 4);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t qoff = ((ks >> 2) * kQHalf + (ks & 3) * 32) >> 4;
      const uint32_t koff = ((ks >> 2) * kKVHalf + (ks & 3) * 32) >> 4;
      umma_ss(tmem + st * 64, qdesc + qoff, kdesc + koff, idesc_qk, ks > 0);
    }
    umma_commit(&bars->s_full[st]);
    umma_commit(&bars->k_empty[st]);
  }
  return true;
}

template <int D>
__device__ bool extend_mma_pv(Bars* bars, uint32_t sb, uint32_t tmem, const Work& w) {
  using C = Cfg<D>;
  constexpr uint32_t idesc_pv = umma_idesc_bf16(kBM, D, true);
  const uint64_t vdesc0 = smem_desc_sw128(sb + C::kOffV, kKVHalf, 1024);
  for (int j = 0; j < w.n_tiles; ++j) {
    const int st = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    if (!mbar_wait(&bars->p_full[st], ph)) return false;
    if (!mbar_wait(&bars->v_full[st], ph)) return false;
    tc_fence_after();
    const uint64_t vdesc = vdesc0 + ((st * C::kKVStage) >> 4);
#pragma unroll
    for (int ks = 0; ks < kBN / 16; ++ks) {
      // P of positions [16ks, 16ks+16): its half's columns of the tile's S buffer, bf16 pairs.
      // V rows [16ks, 16ks+16) as one MN-major operand of N = D; its 64-dim halves are kKVHalf
      // apart.
      const uint32_t pa = tmem + st * 64 + (ks >> 1) * 32 + (ks & 1) * 8;
      umma_ts(tmem + kColO, pa, vdesc + ((ks * 2048) >> 4), idesc_pv, j > 0 || ks > 0);
    }
    umma_commit(&bars->v_empty[st]);
    umma_commit(&bars->s_free[st]);  // P (in the S buffer) consumed; also marks this PV done
  }
  return true;
}

// Packed pairs of fp32 (sm_100 family): {lo, hi} in one 64-bit register pair.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void split_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// acc + (float)(low or high bf16 half of v), one rounding: the sm_100 family's mixed-precision add
__device__ __forceinline__ float add_bf16_lo(uint32_t v, float acc) {
  float r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
      : "=f"(r) : "r"(v), "f"(acc));
  return r;
}
__device__ __forceinline__ float add_bf16_hi(uint32_t v, float acc) {
  float r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
      : "=f"(r) : "r"(v), "f"(acc));
  return r;
}

// max of three (the sm_100 family's three-input max.f32)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max of 32 values in 16 three-input maxima: 32 -> 11 -> 4 -> 1
__device__ __forceinline__ float max32(const float (&v)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]);
  const float b2 = max3f(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return fmaxf(max3f(b0, b1, b2), b3);
}

// Softmax with one thread per row of the tile (four warps, one per TMEM lane quadrant): the
// thread reads all 64 scores of its row, so the row max needs no exchange between warps.
template <int D>
__device__ void extend_softmax(const ExtendArgs& a, uint8_t* smem, Bars* bars, uint32_t tmem,
                               const Work& w) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;       // TMEM lane quadrant this warp may access
  const int r = wq * 32 + lane;  // tile row == TMEM lane
  const int tid = (warp - 2) * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16);
  const int G = a.group;
  const int rt = a.log2_group >= 0 ? r >> a.log2_group : r / G;  // the row's token in the tile
  const int tok = w.t0 + rt;
  const int g = r - rt * G;
  const bool valid = r < a.rows_used && tok < w.E;
  const int limit = min(w.mask0 + tok, w.L - 1);        // last visible KV position of this row
  const int min_limit = min(w.mask0 + w.t0, w.L - 1);  // smallest limit over the tile's rows
  const bool pos_scale = a.scale_log2 > 0.f;
  const float sc = pos_scale ? a.scale_log2 : 1.f;
  float m_used = -INFINITY;  // running max of the scaled (log2) scores
  float l = 0.f;             // running sum of the probabilities (for the LSE)
  float lr = 0.f;            // ... of the probabilities as rounded to bf16 for the PV MMA (for O)
  bool ok = true;

  for (int j = 0; j < w.n_tiles; ++j) {
    const int st = j & 1;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[st], (j >> 1) & 1));
    if (!ok) break;
    tc_fence_after();
    float s0[32], s1[32];  // the row's scores, positions [0, 32) and [32, 64) of the tile
    tmem_ld32(taddr + st * 64, s0);
    tmem_ld32(taddr + st * 64 + 32, s1);
    tmem_wait_ld();
    const int pos0 = j * kBN;
    if (!pos_scale) {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s0[c] *= a.scale_log2;
        s1[c] *= a.scale_log2;
      }
    }
    if (pos0 + kBN - 1 > min_limit) {  // the causal diagonal crosses this tile
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s0[c] = (pos0 + c <= limit) ? s0[c] : -INFINITY;
        s1[c] = (pos0 + 32 + c <= limit) ? s1[c] : -INFINITY;
      }
    }
    const float mx = fmaxf(max32(s0), max32(s1)) * sc;
    const float m_new = fmaxf(m_used, mx);
    const bool resc = m_new > m_used + 8.f;  // always true on the first tile (m_used = -inf)
    const float m_ref = resc ? m_new : m_used;
    const float corr = resc ? ex2(m_used - m_ref) : 1.f;
    const uint64_t sc2 = f32x2(sc, sc), nm2 = f32x2(-m_ref, -m_ref);
    float tot = 0.f, rtot = 0.f;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float(&sv)[32] = hf ? s1 : s0;
      uint32_t pk[16];
      uint64_t acc_a = f32x2(0.f, 0.f), acc_b = f32x2(0.f, 0.f);
      float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        float x0, x1, x2, x3;
        split_f32x2(fma_f32x2(f32x2(sv[2 * c], sv[2 * c + 1]), sc2, nm2), x0, x1);
        split_f32x2(fma_f32x2(f32x2(sv[2 * c + 2], sv[2 * c + 3]), sc2, nm2), x2, x3);
        const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
        acc_a = add_f32x2(acc_a, f32x2(p0, p1));
        acc_b = add_f32x2(acc_b, f32x2(p2, p3));
        pk[c] = pack_bf16x2(p0, p1);
        pk[c + 1] = pack_bf16x2(p2, p3);
        rs0 = add_bf16_lo(pk[c], rs0);
        rs1 = add_bf16_hi(pk[c], rs1);
        rs2 = add_bf16_lo(pk[c + 1], rs2);
        rs3 = add_bf16_hi(pk[c + 1], rs3);
      }
      float e0, e1;
      split_f32x2(add_f32x2(acc_a, acc_b), e0, e1);
      tot += e0 + e1;
      rtot += (rs0 + rs1) + (rs2 + rs3);
      // P (bf16 pairs) over the first 16 columns of each 32-column half of the S buffer, the
      // layout the PV MMA reads
      tmem_st16(taddr + st * 64 + hf * 32, pk);
    }
    l = l * corr + tot;
    lr = lr * corr + rtot;
    m_used = m_ref;

    if (j > 0 && __any_sync(0xffffffffu, resc)) {
      // O is rescaled only after the previous tile's PV is done
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_free[(j - 1) & 1], ((j - 1) >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        const uint32_t oc = taddr + kColO + ch * 32;
        tmem_ld32(oc, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= corr;
        tmem_st32(oc, o);
      }
    }
    tmem_wait_st();
    if (j == w.n_tiles - 1 && w.kv_end < pos0 + kBN) {
      // V rows past the last needed position: zero them so that P = 0 times V stays 0
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (j >> 1) & 1));
      if (!ok) break;
      const int r0 = w.kv_end - pos0;
      const int nchunks = (kBN - r0) * 8 * C::kHalves;  // rows x 16-byte chunks x halves
      uint8_t* vb = smem + C::kOffV + st * C::kKVStage;
      for (int idx = tid; idx < nchunks; idx += kSoftmaxWarps * 32) {
        const int half = idx % C::kHalves, rc = idx / C::kHalves;
        const int row = r0 + (rc >> 3), ch = rc & 7;
        *reinterpret_cast<uint4*>(vb + half * kKVHalf + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->p_full[st]);
  }

  if (ok) {  // the last PV is done
    const int jl = w.n_tiles - 1;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_free[jl & 1], (jl >> 1) & 1));
  }
  if (!ok) {
    if (lane == 0) {
      report(a.err_word, PKV_DEVERR_TIMEOUT);
      bars->epi_skip = 1;
    }
    return;
  }
  // the row's normaliser for the epilogue, which all eight warps share
  reinterpret_cast<float*>(smem + C::kOffInv)[r] = 1.f / lr;
  if (valid && a.lse)
    a.lse[(int64_t)(w.qo0 + tok) * a.num_q_heads + (int64_t)w.h * G + g] = (m_used + log2f(l)) * kLn2;
}

// Epilogue, by all eight warps once the last PV is done: the normalised O tile goes to shared
// memory in the layout of the Q tile's TMA boxes (64-dim halves of 128-byte rows, 16-byte chunk c
// of row r at chunk c ^ (r % 8)), over the Q buffer, which every QK has finished with.  Warp w
// reads TMEM lane quadrant w % 4: the softmax warps read and stage the first 64 dims of their
// rows, the producer and MMA warps (one per quadrant) the second 64, so each thread converts half
// a row.  A full tile then leaves by two TMA stores issued by one thread; the last, partial tile
// of a request (whose box would reach into the next request's rows) is copied out by all threads
// with coalesced 16-byte stores.
template <int D>
__device__ void extend_epilogue(const ExtendArgs& a, uint8_t* smem, uint32_t tmem, const Work& w) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const bool softmax_warp = warp >= 2 && warp < 2 + kSoftmaxWarps;
  const int G = a.group;
  uint8_t* stage = smem + C::kOffQ;
  tc_fence_after();
  if (softmax_warp || C::kHalves == 2) {
    const int hf = softmax_warp ? 0 : 1;
    const float inv = reinterpret_cast<const float*>(smem + C::kOffInv)[r];
    const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16) + kColO + hf * 64;
    float o0[32], o1[32];
    tmem_ld32(taddr, o0);
    tmem_ld32(taddr + 32, o1);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float(&o)[32] = q < 4 ? o0 : o1;
      const int e = (q & 3) * 8;
      *reinterpret_cast<uint4*>(stage + hf * kQHalf + r * 128 + ((q ^ (r & 7)) << 4)) =
          make_uint4(pack_bf16x2(o[e] * inv, o[e + 1] * inv), pack_bf16x2(o[e + 2] * inv, o[e + 3] * inv),
                     pack_bf16x2(o[e + 4] * inv, o[e + 5] * inv), pack_bf16x2(o[e + 6] * inv, o[e + 7] * inv));
    }
  }
  fence_proxy_async_smem();  // the staged tile, before the TMA engine reads it
  __syncthreads();
  if (w.t0 + a.tokens_per_tile <= w.E) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_store_3d(&a.tm_o, hf * 64, w.h * G, w.qo0 + w.t0, smem_u32(stage + hf * kQHalf));
      bulk_commit_group();
      bulk_wait_group_read0();  // shared memory may be released once the stores have read it
    }
  } else {
    constexpr int kCh = C::kChunks;
#pragma unroll
    for (int k = 0; k < kBM * kCh / kThreads; ++k) {
      const int i = threadIdx.x + k * kThreads;
      const int row = i / kCh, c = i % kCh;
      const int tr = a.log2_group >= 0 ? row >> a.log2_group : row / G;
      const int t = w.t0 + tr;
      if (row < a.rows_used && t < w.E) {
        const int64_t orow = (int64_t)(w.qo0 + t) * a.num_q_heads + (int64_t)w.h * G + (row - tr * G);
        reinterpret_cast<uint4*>(a.out + orow * D)[c] = *reinterpret_cast<const uint4*>(
            stage + (c >> 3) * kQHalf + row * 128 + (((c & 7) ^ (row & 7)) << 4));
      }
    }
  }
}

// The request that is z-th in the order "longest KV first, ties by index" (the order kernel's
// order), computed by each warp for batches of up to 32 requests: lane i loads request i's
// metadata and counts the requests that come before it, and the z-th request's metadata is then
// taken from its lane.  Saves the order kernel's launch and a round of dependent loads.
template <bool kCausal>
__device__ __forceinline__ void rank_request(const ExtendArgs& a, int z, Work& w) {
  const int lane = threadIdx.x & 31;
  Work mine{};
  int64_t len = -1;  // lanes past the batch sort last
  if (lane < a.batch) {
    load_request<kCausal>(a, lane, mine);
    len = max(0, mine.P);
    if (kCausal) len += max(0, mine.E);
  }
  int rank = 0;
  for (int j = 0; j < a.batch; ++j) {
    const int64_t lj = __shfl_sync(0xffffffffu, len, j);
    rank += (lj > len || (lj == len && j < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < a.batch && rank == z);
  if (!hit) {  // not reached: the ranks of the batch are a permutation of the grid's z range
    w.b = z;
    load_request<kCausal>(a, z, w);
    return;
  }
  const int src = __ffs(hit) - 1;
  w.b = src;
  w.q0 = __shfl_sync(0xffffffffu, mine.q0, src);
  w.qo0 = __shfl_sync(0xffffffffu, mine.qo0, src);
  w.E = __shfl_sync(0xffffffffu, mine.E, src);
  w.P = __shfl_sync(0xffffffffu, mine.P, src);
  w.p0 = __shfl_sync(0xffffffffu, mine.p0, src);
  w.np = __shfl_sync(0xffffffffu, mine.np, src);
}

// The compact grid of a ranked batch: blockIdx.y enumerates the Q tiles of all requests, the
// requests in the ranked order and each request's tiles last first (most KV first), with no CTA
// for the rows a short request does not have.  Lane i loads request i's metadata and its tile
// count T_i and sums the counts of the requests ranked before it; this CTA's request is the one
// whose range [before, before + T) holds tile index i.  False: no tile left for this CTA.  The
// first CTA reports a request with a negative row count or more rows than max_tiles tiles hold
// (those rows stay unwritten, as with the full grid).
__device__ __forceinline__ bool locate_tile(const ExtendArgs& a, int i, Work& w, bool& first_of_request) {
  const int lane = threadIdx.x & 31;
  Work mine{};
  int64_t len = -1;
  int T = 0;
  if (lane < a.batch) {
    load_request<true>(a, lane, mine);
    len = (int64_t)max(0, mine.P) + max(0, mine.E);
    T = min((max(0, mine.E) + a.tokens_per_tile - 1) / a.tokens_per_tile, a.max_tiles);
  }
  int before = 0, total = 0;
  for (int j = 0; j < a.batch; ++j) {
    const int64_t lj = __shfl_sync(0xffffffffu, len, j);
    const int tj = __shfl_sync(0xffffffffu, T, j);
    before += (lj > len || (lj == len && j < lane)) ? tj : 0;
    total += tj;
  }
  if (i == 0 && blockIdx.x == 0) {
    const unsigned bad = __ballot_sync(0xffffffffu, lane < a.batch &&
                                                        (mine.E < 0 || mine.E > (int64_t)a.max_tiles * a.tokens_per_tile));
    if (threadIdx.x == 0 && (bad || total > (int)gridDim.y)) report(a.err_word, PKV_DEVERR_LENGTH);
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < a.batch && i >= before && i < before + T);
  if (!hit) return false;
  const int src = __ffs(hit) - 1;
  w.b = src;
  w.q0 = __shfl_sync(0xffffffffu, mine.q0, src);
  w.qo0 = __shfl_sync(0xffffffffu, mine.qo0, src);
  w.E = __shfl_sync(0xffffffffu, mine.E, src);
  w.P = __shfl_sync(0xffffffffu, mine.P, src);
  w.p0 = __shfl_sync(0xffffffffu, mine.p0, src);
  w.np = __shfl_sync(0xffffffffu, mine.np, src);
  const int k = i - __shfl_sync(0xffffffffu, before, src);  // k-th tile from the request's end
  w.t0 = (__shfl_sync(0xffffffffu, T, src) - 1 - k) * a.tokens_per_tile;
  first_of_request = w.t0 == 0;
  return true;
}

template <bool kCausal, int D, bool kRows>
__global__ void __launch_bounds__(kThreads, 2) paged_extend_kernel(const __grid_constant__ ExtendArgs a) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Work w;
  bool reporter;  // the CTA that reports its request's argument errors (one per request)
  if (kCausal && a.compact) {
    w.h = blockIdx.x;
    if (!locate_tile(a, (int)blockIdx.y, w, reporter)) return;
    reporter = reporter && blockIdx.x == 0;
  } else {
    // later tiles of a request attend over more positions: launch them first
    w.t0 = (gridDim.x - 1 - blockIdx.x) * a.tokens_per_tile;
    w.h = blockIdx.y;
    if (a.rank_inline) {
      rank_request<kCausal>(a, (int)blockIdx.z, w);
    } else {
      w.b = a.order ? __ldg(a.order + blockIdx.z) : (int)blockIdx.z;
      load_request<kCausal>(a, w.b, w);
    }
    reporter = blockIdx.x == gridDim.x - 1 && blockIdx.y == 0;
    // the grid covers gridDim.x * tokens_per_tile rows of each request (max_extend_len, or the
    // largest part): a request with more rows, or a negative count, is reported once, by the CTA
    // of its first tile, and its rows past the grid stay unwritten
    if (reporter && threadIdx.x == 0 && (w.E < 0 || w.E > (int)gridDim.x * a.tokens_per_tile))
      report(a.err_word, PKV_DEVERR_LENGTH);
    if (w.t0 >= w.E) return;  // uniform: this tile has no rows
  }
  if (w.q0 < 0 || w.qo0 < 0 || w.q0 > a.num_q_rows - w.E || w.qo0 > a.num_out_rows - w.E) {
    if (threadIdx.x == 0 && reporter) report(a.err_word, PKV_DEVERR_ROW_OOB);
    return;
  }
  const int P = w.P;
  if (kCausal) {
    w.mask0 = P;
    w.L = P + w.E;
    w.kv_end = P + min(w.t0 + a.tokens_per_tile, w.E);
  } else {
    // every row sees the part's whole KV
    w.L = max(P, 0);
    w.mask0 = w.L;
    w.kv_end = w.L;
    if (P < 0 && threadIdx.x == 0 && reporter) report(a.err_word, PKV_DEVERR_LENGTH);
  }
  w.n_tiles = (w.kv_end + kBN - 1) / kBN;
  if (w.n_tiles == 0) {  // a part with no KV: o = 0, lse = -inf (uniform over the CTA)
    const int G = a.group;
    const int rows = min(a.tokens_per_tile, w.E - w.t0) * G;
    for (int i = threadIdx.x; i < rows * (D / 8); i += kThreads) {
      const int row = i / (D / 8), c = i % (D / 8);
      const int64_t orow = (int64_t)(w.qo0 + w.t0 + row / G) * a.num_q_heads + (int64_t)w.h * G + row % G;
      reinterpret_cast<uint4*>(a.out + orow * D)[c] = make_uint4(0u, 0u, 0u, 0u);
      if (c == 0 && a.lse) a.lse[orow] = -INFINITY;
    }
    return;
  }
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.err_word, PKV_DEVERR_INTERNAL);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 1);
    }
    mbar_init(&bars->qk_done, 1);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->p_full[0], kSoftmaxWarps);
    mbar_init(&bars->p_full[1], kSoftmaxWarps);
    bars->epi_skip = 0;
    fence_mbar_init();
    prefetch_tmap(&a.tm_k);
    prefetch_tmap(&a.tm_v);
    prefetch_tmap(&a.tm_o);
    // Q first, before the rest of the set-up: one box per 64-dim half, [64 dims x G heads x
    // tokens_per_tile tokens], rows_used rows
    mbar_arrive_expect_tx(&bars->q_full, C::kHalves * a.rows_used * 128);
#pragma unroll
    for (int hf = 0; hf < C::kHalves; ++hf)
      tma_load_3d(sb + C::kOffQ + hf * kQHalf, &a.tm_q, hf * 64, w.h * a.group, w.q0 + w.t0, &bars->q_full);
  }
  // the producers' page-list window, loading while TMEM is allocated and the CTA synchronises
  PageWindow pw{-1, -1};
  if (!kRows && (warp == 0 || warp == kVWarp)) pw = load_page_window(a, w);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0 || warp == kVWarp) {
    if (kRows)
      extend_producer_rows<D>(a, sb, bars, w, warp == 0 ? 0 : 1);
    else
      extend_producer<D>(a, sb, bars, w, warp == 0 ? 0 : 1, pw);
  } else if (warp == 1) {
    if (lane == 0) {
      if (!extend_mma_qk<D>(a, sb, bars, tmem, w)) report(a.err_word, PKV_DEVERR_TIMEOUT);
      // its MMAs have completed before TMEM is released (immediate on the normal path)
      umma_commit(&bars->qk_done);
      if (!mbar_wait(&bars->qk_done, 0)) report(a.err_word, PKV_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kPVWarp) {
    if (lane == 0) {
      if (!extend_mma_pv<D>(bars, sb, tmem, w)) report(a.err_word, PKV_DEVERR_TIMEOUT);
      umma_commit(&bars->pv_done);
      if (!mbar_wait(&bars->pv_done, 0)) report(a.err_word, PKV_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    extend_softmax<D>(a, smem, bars, tmem, w);
  }
  tc_fence_before();
  __syncthreads();  // every warp is done with its stream; O is complete unless a wait gave up
  if (!bars->epi_skip) extend_epilogue<D>(a, smem, tmem, w);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Requests ordered by KV length (prefix + new tokens; a shared-prefix part's whole KV when
// qo_indptr is null), longest first and ties by index, so that the grid dispatches the CTAs with
// the most work first and the last wave holds short ones: a bitonic sort of (length, index) keys
// in shared memory by one CTA.  n is a power of two >= B.
constexpr int kMaxOrdered = 4096;
constexpr int kInlineRanked = 32;

__global__ void __launch_bounds__(1024) extend_order_kernel(const int32_t* __restrict__ qo_indptr,
                                                            const int32_t* __restrict__ prefix_lens,
                                                            int32_t B, int32_t n, int32_t* __restrict__ order) {
  __shared__ unsigned long long key[kMaxOrdered];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    unsigned long long k = 0;  // padding sorts last
    if (i < B) {
      const int64_t L = (int64_t)max(0, __ldg(prefix_lens + i)) +
                        (qo_indptr ? max(0, __ldg(qo_indptr + i + 1) - __ldg(qo_indptr + i)) : 0);
      const unsigned long long len = (unsigned long long)min(L, (int64_t)0x7fffffff);
      k = (len << 32) | (0xffffffffull - (unsigned)i);  // larger first; equal lengths by index
    }
    key[i] = k;
  }
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = key[i], y = key[ixj];
          const bool descending = (i & k) == 0;
          if (descending ? x < y : x > y) {
            key[i] = y;
            key[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < B; i += blockDim.x)
    order[i] = (int32_t)(0xffffffffull - (key[i] & 0xffffffffull));
}

// ---------------------------------------------------------------------------------------------
// Host
// ---------------------------------------------------------------------------------------------
int log2_exact(int x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

}  // namespace

extern "C" {

size_t pkv_extend_workspace_size(int32_t batch_size, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_extend_len) {
  (void)num_q_heads;
  (void)num_kv_heads;
  (void)head_dim;
  (void)max_extend_len;
  // the request order (int32 per request) when the batch is small enough to sort in one CTA
  // (batches of up to kInlineRanked requests are ranked inside the extend kernel: no workspace)
  if (batch_size <= kInlineRanked || batch_size > kMaxOrdered) return 0;
  return ((size_t)batch_size * 4 + 255) & ~(size_t)255;
}

}  // extern "C"

namespace {

template <bool kCausal, int D, bool kRows>
pkv_status launch_kernel(const ExtendArgs& a, dim3 grid, cudaStream_t stream) {
  constexpr uint32_t smem = Cfg<D>::kSmemBytes;
  // whether this instance's dynamic shared-memory limit was raised on this device (any host thread)
  static std::atomic<bool> configured[64];
  const int dev = pkv_host::current_device();
  if (dev < 0) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(paged_extend_kernel<kCausal, D, kRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_relaxed);
  }
  paged_extend_kernel<kCausal, D, kRows><<<grid, kThreads, smem, stream>>>(a);
  return pkv_host::launch_status();
}

// The launch shared by the extend (causal) and the shared-prefix parts (causal == 0):
// the host checks, the tensor maps, the request order and the kernel.
pkv_status launch_extend(const pkv_pool* pool, const void* q, int32_t num_q_rows, int32_t num_out_rows,
                         const int32_t* qo_indptr, const int32_t* q_start, const int32_t* o_start,
                         const int32_t* q_len, int causal, int32_t batch_size, int32_t num_q_heads,
                         const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_lens,
                         int32_t max_rows, float sm_scale, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, uint32_t* err_word, void* stream) {
  if (!pkv_host::valid_pool(pool) || batch_size < 0 || num_q_heads <= 0 || num_q_rows < 0 ||
      num_out_rows < 0 || max_rows < 0)
    return PKV_ERR_INVALID_ARG;
  if (batch_size == 0 || num_q_rows == 0 || num_out_rows == 0 || max_rows == 0) return PKV_OK;
  if (!q || !kv_indptr || !kv_indices || !kv_lens || !out) return PKV_ERR_INVALID_ARG;
  if (causal ? !qo_indptr : (!q_start || !o_start || !q_len)) return PKV_ERR_INVALID_ARG;
  const size_t ws_need = pkv_extend_workspace_size(batch_size, num_q_heads, pool->num_kv_heads,
                                                   pool->head_dim, max_rows);
  if (ws_need > 0 && (!workspace || workspace_bytes < ws_need)) return PKV_ERR_WORKSPACE;
  if (ws_need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PKV_ERR_INVALID_ARG;
  if (!pkv_host::aligned16(q) || !pkv_host::aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int D = pool->head_dim;
  if (D != 64 && D != 128) return PKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / pool->num_kv_heads;
  if (G > 16) return PKV_ERR_UNSUPPORTED;
  // page boxes of at least 8 rows keep every TMA destination on a 1024-byte swizzle atom; other
  // page sizes take the row-copy producer
  const int lps = log2_exact(pool->page_size);
  const bool rows_path = lps < 3;
  if (pool->num_pages * (int64_t)pool->page_size > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (batch_size > 65535 || pool->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;

  ExtendArgs a;
  const int tpt = kBM / G;
  const uint64_t Hq = num_q_heads, Hkv = pool->num_kv_heads;
  const uint64_t rows = (uint64_t)pool->num_pages * pool->page_size;
  const uint32_t R = rows_path ? 8 : (pool->page_size < kBN ? pool->page_size : kBN);  // TMA box rows
  const uint64_t Db = (uint64_t)D * 2;
  if (!pkv_host::encode_tmap_3d(&a.tm_q, q, D, Hq, (uint64_t)num_q_rows, Db, Hq * Db, 64, G, tpt) ||
      !pkv_host::encode_tmap_3d(&a.tm_o, out, D, Hq, (uint64_t)num_out_rows, Db, Hq * Db, 64, G, tpt) ||
      !pkv_host::encode_tmap_3d(&a.tm_k, pool->k, D, Hkv, rows, Db, Hkv * Db, 64, 1, R) ||
      !pkv_host::encode_tmap_3d(&a.tm_v, pool->v, D, Hkv, rows, Db, Hkv * Db, 64, 1, R))
    return PKV_ERR_CUDA;
  a.qo_indptr = qo_indptr;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.prefix_lens = kv_lens;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  a.err_word = err_word;
  a.num_pages = pool->num_pages;
  a.page_size = pool->page_size;
  a.log2_ps = lps;
  a.k_pool = (const __nv_bfloat16*)pool->k;
  a.v_pool = (const __nv_bfloat16*)pool->v;
  a.num_kv_heads = pool->num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.group = G;
  a.rows_used = G * tpt;
  a.log2_group = log2_exact(G);
  a.tokens_per_tile = tpt;
  a.scale_log2 = sm_scale * kLog2e;
  a.order = nullptr;
  a.rank_inline = batch_size <= kInlineRanked ? 1 : 0;
  const int tiles = (max_rows + tpt - 1) / tpt;
  // the compact grid needs no more CTAs per kv head than the batch's Q tiles can number:
  // sum_b ceil(E_b / tpt) < num_q_rows / tpt + batch
  const int64_t compact_tiles =
      std::min<int64_t>((int64_t)tiles * batch_size, ((int64_t)num_q_rows + tpt - 1) / tpt + batch_size);
  a.compact = causal && a.rank_inline && compact_tiles <= 65535 ? 1 : 0;
  a.max_tiles = tiles;
  a.batch = batch_size;
  a.q_start = q_start;
  a.o_start = o_start;
  a.q_len = q_len;
  a.num_q_rows = num_q_rows;
  a.num_out_rows = num_out_rows;
  if (ws_need > 0) {
    int n = 1;
    while (n < batch_size) n <<= 1;
    extend_order_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(causal ? qo_indptr : nullptr, kv_lens,
                                                              batch_size, n, (int32_t*)workspace);
    const pkv_status st = pkv_host::launch_status();
    if (st != PKV_OK) return st;
    a.order = (const int32_t*)workspace;
  }

  const dim3 grid = a.compact ? dim3(pool->num_kv_heads, (unsigned)compact_tiles, 1)
                              : dim3(tiles, pool->num_kv_heads, batch_size);
  cudaStream_t st = (cudaStream_t)stream;
  if (rows_path) {
    if (D == 128)
      return causal ? launch_kernel<true, 128, true>(a, grid, st) : launch_kernel<false, 128, true>(a, grid, st);
    return causal ? launch_kernel<true, 64, true>(a, grid, st) : launch_kernel<false, 64, true>(a, grid, st);
  }
  if (D == 128)
    return causal ? launch_kernel<true, 128, false>(a, grid, st) : launch_kernel<false, 128, false>(a, grid, st);
  return causal ? launch_kernel<true, 64, false>(a, grid, st) : launch_kernel<false, 64, false>(a, grid, st);
}

}  // namespace

extern "C" {

pkv_status pkv_paged_extend(const pkv_pool* pool, const void* q, int32_t num_q_tokens,
                            const int32_t* qo_indptr, int32_t batch_size, int32_t num_q_heads,
                            const int32_t* kv_indptr, const int32_t* kv_indices,
                            const int32_t* prefix_lens, int32_t max_extend_len, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            uint32_t* err_word, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_extend");
  return launch_extend(pool, q, num_q_tokens, num_q_tokens, qo_indptr, nullptr, nullptr, nullptr, 1,
                       batch_size, num_q_heads, kv_indptr, kv_indices, prefix_lens, max_extend_len,
                       sm_scale, out, lse, workspace, workspace_bytes, err_word, stream);
}

size_t pkv_shared_prefix_workspace_size(int32_t num_parts, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t max_part_rows) {
  return pkv_extend_workspace_size(num_parts, num_q_heads, num_kv_heads, head_dim, max_part_rows);
}

pkv_status pkv_shared_prefix_attention(const pkv_pool* pool, const void* q, int32_t num_q_rows,
                                       const int32_t* q_start, const int32_t* q_len,
                                       const int32_t* o_start, int32_t num_parts, int32_t num_q_heads,
                                       const int32_t* kv_indptr, const int32_t* kv_indices,
                                       const int32_t* kv_lens, int32_t max_part_rows, float sm_scale,
                                       void* o_part, float* lse_part, int32_t num_out_rows,
                                       void* workspace, size_t workspace_bytes, uint32_t* err_word,
                                       void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_shared_prefix_attention");
  return launch_extend(pool, q, num_q_rows, num_out_rows, nullptr, q_start, o_start, q_len, 0,
                       num_parts, num_q_heads, kv_indptr, kv_indices, kv_lens, max_part_rows, sm_scale,
                       o_part, lse_part, workspace, workspace_bytes, err_word, stream);
}

}  // extern "C"
