// Paged decode attention (one query per request) and the split-KV log-sum-exp merge.
//
// What it computes: for request b and query head h, attention of q[b,h] over the request's
// kv_lens[b] KV positions, gathered in place from the paged pool through the CSR page list
// (nanoSGLang README, "Ablation": paged attention with zero-copy KV; Mini-SGLang README,
// "Reference Attention Backends": paged KV gather, GQA via repeat_interleave, online softmax in
// the Triton decode kernel).  Long requests are split and merged by log-sum-exp (flash-decoding).
//
// Design for GB300 (HBM-bound: ~2-8 flop per KV byte):
//  * Persistent grid, one CTA per SM.  The KV of all (request, KV-head-group) units, cut into
//    16-token slices counted from each unit's first position, forms one stream; every CTA takes an
//    equal contiguous share of slices, so work is balanced whatever the length mix.  A unit cut by
//    a share boundary leaves one partial per CTA that touched it, merged by a second kernel.  A CTA
//    covers HC KV heads, so one token row of the CTA is a single contiguous HC*D*2-byte run.
//  * One producer warp walks the share and fills a ring of shared-memory stages, completion
//    counted in bytes on mbarriers.  When the page size is a multiple of 16 a 16-token slice lies
//    in one page and is fetched by TMA as one 3-D box per 64-dim half, [64 dims x 16 rows x HC
//    heads] with 128-byte swizzle: each head's slice lands as its own 2 KB block whose rows are
//    swizzled, so the warps' ldmatrix reads are conflict free.  Other page sizes use one
//    cp.async.bulk per token row, into rows padded to a conflict-free stride.
//  * Consumer warps (one per KV head, W per head when HC < 8) take 16-token slices.  Scores are
//    computed transposed, S^T = K Q^T, with m16n8k16 bf16 MMAs (tokens fill M=16, the G query
//    heads of the group fill N=8, so nothing is padded to 16 heads); the online softmax keeps a
//    running max and sum in fp32 per head; P^T is turned into the B operand of O^T += V^T P^T by
//    movmatrix.  KV is read exactly once per CTA per token, for all heads of the group.
#include <float.h>

#include <atomic>

#include <mutex>
#include <type_traits>

#include "tc05.cuh"

namespace {

using namespace pkv;

constexpr int kSegFirst = 1;    // first stage of this CTA's segment of the unit
constexpr int kSegLast = 2;     // last stage of the segment
constexpr int kStartsUnit = 4;  // the segment starts at position 0 of the unit
constexpr int kEndsUnit = 8;    // the segment ends at the unit's last position

struct StageHdr {
  int32_t unit;  // -1: no more work
  int32_t b;
  int32_t hg;
  int32_t tok0;
  int32_t ntok;
  int32_t flags;
  int32_t part;
  int32_t pad;
};

struct DecodeArgs {
  CUtensorMap tm_k;  // pool as (dim, row, head), box [64 x 16 x HC]; used when use_tma
  CUtensorMap tm_v;
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int64_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  const __nv_bfloat16* q;
  int32_t batch;
  int32_t num_q_heads;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_lens;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  const int32_t* keep_tokens;  // nullable: positions below keep_tokens[b] evict-last in L2, the rest evict-first
  int32_t* unit_first;
  int32_t* unit_last;
  uint32_t* err_word;
  int32_t HC;            // KV heads per CTA
  int32_t nhg;           // head groups = num_kv_heads / HC
  int32_t W;             // consumer warps per KV head
  int32_t group;         // query heads per KV head
  int32_t row_stride;    // shared-memory bytes per token row (row-copy layout)
  int32_t stage_tokens;  // tokens per stage = 16 * W
  int32_t num_stages;
  int32_t num_parts;     // partial slots in the workspace
  uint32_t kv_region;    // bytes of the K (or V) part of one stage
};

constexpr int kMaxStages = 8;

template <int D, int NT>
struct Consumer {
  static constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of O^T
  // floats per lane exchanged when W > 1 warps share a head: m, l and O^T fragments
  static constexpr int kMergeFloats = 4 * NT + KS * NT * 4;
};

// ---------------------------------------------------------------------------------------------
// Producer: walk the CTA's share of the slice stream and fill stages.
// ---------------------------------------------------------------------------------------------
template <int D, bool TMA>
__device__ void decode_producer(const DecodeArgs& a, uint8_t* stages, StageHdr* hdr,
                                uint64_t* full, uint64_t* empty) {
  const int lane = threadIdx.x & 31;
  const int NS = a.num_stages, Ts = a.stage_tokens, RS = a.row_stride, W = a.W;
  const int nhg = a.nhg;
  const int ps = a.page_size;
  const uint32_t RB = (uint32_t)a.HC * D * 2;
  const int64_t row_elems = (int64_t)a.num_kv_heads * D;
  const uint32_t region = a.kv_region;
  // bytes one 16-token slice brings in (K and V) on the TMA path
  const uint32_t slice_bytes = (uint32_t)(D / 64) * a.HC * 16 * 128 * 2;
  // Page indices come from a register window of 96 consecutive page-list entries (three 32-lane
  // slices).  A stage reads only the first 64; the third slice is loaded when the window moves,
  // 32 pages before any stage can need it, so the copies of a stage never wait on a global load
  // even when a stage spans 16 pages (page size 1).  Usable when one stage spans at most 33 pages.
  const bool windowed = (Ts - 1) / ps + 2 <= 32;

  int64_t sumS = 0;  // 16-token slices over all requests
  for (int i = lane; i < a.batch; i += 32) {
    // the walk below reads the page-list offsets next: bring them to L2 meanwhile
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.kv_indptr + i));
    sumS += (max(0, __ldg(a.kv_lens + i)) + 15) / 16;
  }
  sumS = warp_sum(sumS);
  const int64_t T = sumS * nhg;
  int64_t share = (T + gridDim.x - 1) / gridDim.x;
  if (share < 1) share = 1;
  const int64_t c0 = (int64_t)blockIdx.x * share;
  const int64_t c1 = min(T, c0 + share);

  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;

  int32_t cur_p0 = 0, cur_p1 = 0;  // page list of the request being streamed
  int win_b = -1, wbase = 0;
  int32_t w0 = -1, w1 = -1, w2 = -1;

  auto entry = [&](int pidx) -> int32_t {  // page-list entry pidx of the current request; -1 past its end
    const int64_t s = (int64_t)cur_p0 + pidx;
    return (pidx >= 0 && s < cur_p1) ? __ldg(a.kv_indices + s) : -1;
  };
  auto window_page = [&](int pidx) -> int32_t {  // all lanes must call; pidx - wbase < 64
    const int k = pidx - wbase;
    const int32_t v0 = __shfl_sync(0xffffffffu, w0, k & 31);
    const int32_t v1 = __shfl_sync(0xffffffffu, w1, k & 31);
    return k < 32 ? v0 : v1;
  };

  // L2 policies of the keep hint (made once; unused without a hint)
  const uint64_t pol_keep = policy_evict_last(), pol_stream = policy_evict_first();

  int nissued = 0;  // stages handed to the consumers (copies, or the end marker)
  auto next_stage = [&]() {
    ++nissued;
    if (++stage == NS) {
      stage = 0;
      phase ^= 1;
    }
  };

  auto emit = [&](int unit, int b, int hg, int tok0, int ntok, int flags) -> bool {
    if (unit >= 0 && (flags & kSegFirst)) {
      // the consumers read this unit's queries when its first stage lands: bring them to L2 now
      const int hqu = a.HC * a.group;
      const char* qb = reinterpret_cast<const char*>(a.q + ((int64_t)b * a.num_q_heads + (int64_t)hg * hqu) * D);
      for (int off = lane * 128; off < hqu * D * 2; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + off));
    }
    if (unit >= 0 && windowed) {
      const int first_page = tok0 / ps;
      if (b != win_b || first_page < wbase) {  // new request or restart from its first page
        win_b = b;
        wbase = first_page;
        w0 = entry(wbase + lane);
        w1 = entry(wbase + 32 + lane);
        w2 = entry(wbase + 64 + lane);
      }
      while (first_page >= wbase + 32) {
        w0 = w1;
        w1 = w2;
        wbase += 32;
        w2 = entry(wbase + 64 + lane);
      }
    }
    if (!mbar_wait(&empty[stage], phase ^ 1)) {
      if (lane == 0) report(a.err_word, PKV_DEVERR_TIMEOUT);
      return false;
    }
    if (lane == 0) {
      StageHdr h;
      h.unit = unit;
      h.b = b;
      h.hg = hg;
      h.tok0 = tok0;
      h.ntok = ntok;
      h.flags = flags;
      h.part = blockIdx.x + unit;
      h.pad = 0;
      hdr[stage] = h;
    }
    uint8_t* kst = stages + (size_t)stage * 2 * region;
    uint8_t* vst = kst + region;
    if (unit < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[stage]);
      next_stage();
      return true;
    }
    if constexpr (TMA) {
      // lane s < W fetches slice s of the stage: 16 tokens inside one page
      const int tok = tok0 + 16 * lane;
      const bool in = lane < W && tok < tok0 + ntok;
      const int pidx = tok / ps;
      const int32_t page = windowed ? window_page(pidx) : (in ? entry(pidx) : -1);
      int row = -1;
      uint32_t bad = 0;
      if (in) {
        if ((int64_t)cur_p0 + pidx >= cur_p1)
          bad = PKV_DEVERR_LENGTH;
        else if (page < 0 || page >= a.num_pages)
          bad = PKV_DEVERR_PAGE_OOB;
        else
          row = page * ps + tok % ps;
      }
      if (bad) report(a.err_word, bad);
      const int nload = __popc(__ballot_sync(0xffffffffu, row >= 0));
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)nload * slice_bytes);
      __syncwarp();
      if (row >= 0) {
        const uint32_t slice_off = (uint32_t)lane * a.HC * 2048;
        const uint32_t half_stride = (uint32_t)W * a.HC * 2048;
        if (a.keep_tokens) {
          const uint64_t pol = tok < __ldg(a.keep_tokens + b) ? pol_keep : pol_stream;
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_3d_hint(smem_u32(kst) + hf * half_stride + slice_off, &a.tm_k, hf * 64, row, hg * a.HC,
                             &full[stage], pol);
            tma_load_3d_hint(smem_u32(vst) + hf * half_stride + slice_off, &a.tm_v, hf * 64, row, hg * a.HC,
                             &full[stage], pol);
          }
        } else {
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_3d(smem_u32(kst) + hf * half_stride + slice_off, &a.tm_k, hf * 64, row, hg * a.HC, &full[stage]);
            tma_load_3d(smem_u32(vst) + hf * half_stride + slice_off, &a.tm_v, hf * 64, row, hg * a.HC, &full[stage]);
          }
        }
      }
    } else {
      // up to 4 rows per lane (stage_tokens <= 128), one bulk copy per token row
      int64_t src[4];
      int nvalid = 0;
      uint32_t bad = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = lane + 32 * r;
        const int pos = tok0 + j;
        const int pidx = pos / ps;
        const int32_t page = windowed ? window_page(pidx) : (j < ntok ? entry(pidx) : -1);
        src[r] = -1;
        if (j < ntok) {
          if ((int64_t)cur_p0 + pidx >= cur_p1) {
            bad |= PKV_DEVERR_LENGTH;
          } else if (page < 0 || page >= a.num_pages) {
            bad |= PKV_DEVERR_PAGE_OOB;
          } else {
            src[r] = ((int64_t)page * ps + pos % ps) * row_elems + (int64_t)hg * a.HC * D;
            ++nvalid;
          }
        }
      }
      if (bad) report(a.err_word, bad);
      const int tot = warp_sum(nvalid);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)tot * RB * 2);
      __syncwarp();
      const int keep = a.keep_tokens ? __ldg(a.keep_tokens + b) : 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (src[r] >= 0) {
          const int j = lane + 32 * r;
          if (a.keep_tokens) {
            const uint64_t pol = tok0 + j < keep ? pol_keep : pol_stream;
            bulk_g2s_hint(kst + (size_t)j * RS, a.k_pool + src[r], RB, &full[stage], pol);
            bulk_g2s_hint(vst + (size_t)j * RS, a.v_pool + src[r], RB, &full[stage], pol);
          } else {
            bulk_g2s(kst + (size_t)j * RS, a.k_pool + src[r], RB, &full[stage]);
            bulk_g2s(vst + (size_t)j * RS, a.v_pool + src[r], RB, &full[stage]);
          }
        }
      }
    }
    next_stage();
    return true;
  };

  if (c0 < c1) {
    int64_t base = 0;  // stream offset (in slices) of request b0
    for (int b0 = 0; b0 < a.batch && base < c1 && ok; b0 += 32) {
      const int b = b0 + lane;
      const bool in = b < a.batch;
      const int64_t L = in ? (int64_t)max(0, __ldg(a.kv_lens + b)) : 0;
      const int64_t S = (L + 15) / 16;
      const int32_t ip0 = in ? __ldg(a.kv_indptr + b) : 0;
      const int32_t ip1 = in ? __ldg(a.kv_indptr + b + 1) : 0;
      int64_t incl = S;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int64_t rs = base + nhg * (incl - S);
      const int64_t re = base + nhg * incl;
      uint32_t mask = __ballot_sync(0xffffffffu, in && S > 0 && re > c0 && rs < c1);
      while (mask && ok) {
        const int src_lane = __ffs(mask) - 1;
        mask &= mask - 1;
        const int bb = b0 + src_lane;
        const int64_t Lb = __shfl_sync(0xffffffffu, L, src_lane);
        const int64_t Sb = __shfl_sync(0xffffffffu, S, src_lane);
        const int64_t rsb = __shfl_sync(0xffffffffu, rs, src_lane);
        cur_p0 = __shfl_sync(0xffffffffu, ip0, src_lane);
        cur_p1 = __shfl_sync(0xffffffffu, ip1, src_lane);
        for (int hg = 0; hg < nhg && ok; ++hg) {
          const int64_t us = rsb + (int64_t)hg * Sb, ue = us + Sb;
          const int64_t s0 = max(us, c0), s1 = min(ue, c1);
          if (s0 >= s1) continue;
          const int t0 = (int)(s0 - us) * 16;
          const int t1 = (int)min((s1 - us) * 16, Lb);
          const int unit = bb * nhg + hg;
          for (int t = t0; t < t1 && ok; t += Ts) {
            int flags = 0;
            if (t == t0) flags |= kSegFirst;
            if (t + Ts >= t1) flags |= kSegLast;
            if (s0 == us) flags |= kStartsUnit;
            if (s1 == ue) flags |= kEndsUnit;
            ok = emit(unit, bb, hg, t, min(Ts, t1 - t), flags);
          }
        }
      }
      base += nhg * __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (ok) emit(-1, 0, 0, 0, 0, 0);
  // Wait (bounded) until the copies of the last NS stages issued have landed, so that no copy
  // into this CTA's shared memory is in flight when it exits, also when the consumers gave up on
  // a wait and left.  On the normal path the consumers have already seen every stage complete.
  for (int k = 0; k < min(nissued, NS); ++k) {
    if (--stage < 0) {
      stage = NS - 1;
      phase ^= 1;
    }
    mbar_wait(&full[stage], phase);
  }
}

// ---------------------------------------------------------------------------------------------
// Consumers: 16-token slices of one KV head with its G query heads.
// ---------------------------------------------------------------------------------------------
template <int D, int NT, bool TMA>
__device__ void decode_consumer(const DecodeArgs& a, uint8_t* stages, StageHdr* hdr,
                                uint64_t* full, uint64_t* empty, float* mbuf) {
  constexpr int KS = D / 16;
  constexpr int MF = Consumer<D, NT>::kMergeFloats;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HC = a.HC, W = a.W, G = a.group;
  const int NC = HC * W;
  const int hl = warp % HC;  // KV head within the CTA's group
  const int si = warp / HC;  // slice within a stage
  const int g = lane >> 2, c = lane & 3;
  const int NS = a.num_stages, RS = a.row_stride;
  const uint32_t region = a.kv_region;
  const int HQU = HC * G;  // query heads per unit

  // per-lane ldmatrix addressing.  Row-copy layout: token rows at stride RS, head hl at hl*D*2.
  // TMA layout: [half][slice][head][16 rows][128 B] with the 16-byte chunks of row t XOR-ed by t%8.
  const int mi = lane >> 3, ri = lane & 7;
  const int kt = ri + ((mi & 1) << 3);  // token row this lane addresses for K
  const int vt = ri + ((mi >> 1) << 3);  // ... for V
  uint32_t k_lane_off, v_lane_off;
  const uint32_t half_stride = (uint32_t)W * HC * 2048;
  if (TMA) {
    k_lane_off = (uint32_t)(si * HC * 2048 + hl * 2048 + kt * 128);
    v_lane_off = (uint32_t)(si * HC * 2048 + hl * 2048 + vt * 128);
  } else {
    k_lane_off = (uint32_t)((si * 16 + kt) * RS + hl * D * 2 + ((mi >> 1) << 3) * 2);
    v_lane_off = (uint32_t)((si * 16 + vt) * RS + hl * D * 2 + ((mi & 1) << 3) * 2);
  }
  const uint32_t stages_u32 = smem_u32(stages);

  uint32_t qf[NT][KS][2];
  float o[KS][NT][4];
  float m[NT][2], l[NT][2];

  int stage = 0;
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait(&full[stage], phase)) {
      if (lane == 0) report(a.err_word, PKV_DEVERR_TIMEOUT);
      break;
    }
    const StageHdr h = hdr[stage];
    if (h.unit < 0) break;

    if (h.flags & kSegFirst) {
      // query fragments (B operand of S^T = K Q^T): lane (g, c) holds q[head g][16ks + 2c, +1]
      // and [16ks + 2c + 8, +9]
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + g;
        const bool valid = head < G;
        const __nv_bfloat16* qp =
            a.q + ((int64_t)h.b * a.num_q_heads + (int64_t)(h.hg * HC + hl) * G + head) * D + 2 * c;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qf[nt][ks][0] = valid ? ld_nc_u32(qp + ks * 16) : 0u;
          qf[nt][ks][1] = valid ? ld_nc_u32(qp + ks * 16 + 8) : 0u;
        }
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
      }
    }

    const int nv = min(16, h.ntok - si * 16);
    const uint32_t kb = stages_u32 + (uint32_t)stage * 2 * region;
    const uint32_t vb = kb + region;
    if (nv > 0 && nv < 16) {
      // a partial slice: the rows past the request's end hold unused pool slots (the TMA box
      // brings them, possibly NaN) or whatever shared memory held before (the row copies skip
      // them); zero this head's V rows there so that P = 0 times V stays 0.  K rows there are
      // masked by a select, so their contents never matter.
      uint8_t* vreg = stages + (size_t)stage * 2 * region + region;
      if (TMA) {
        uint8_t* vrow = vreg + si * HC * 2048 + hl * 2048;
        for (int idx = lane; idx < (16 - nv) * 8 * (D / 64); idx += 32) {
          const int hf = idx / ((16 - nv) * 8);
          const int rem = idx - hf * (16 - nv) * 8;
          *reinterpret_cast<uint4*>(vrow + hf * half_stride + (nv + (rem >> 3)) * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        constexpr int kChunks = D * 2 / 16;  // 16-byte chunks of one head's row
        for (int idx = lane; idx < (16 - nv) * kChunks; idx += 32) {
          const int row = si * 16 + nv + idx / kChunks;
          *reinterpret_cast<uint4*>(vreg + (size_t)row * RS + hl * D * 2 + (idx % kChunks) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
    }
    if (nv > 0) {
      float s[NT][4], s2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = s2[nt][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        uint32_t addr;
        if (TMA) {
          const int cc = 2 * (ks & 3) + (mi >> 1);  // 16-byte chunk within the 128-byte row
          addr = kb + (ks >> 2) * half_stride + k_lane_off + ((cc ^ (kt & 7)) << 4);
        } else {
          addr = kb + k_lane_off + ks * 32;
        }
        ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (ks & 1)
            mma_bf16_16816(s2[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
          else
            mma_bf16_16816(s[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
        }
      }
      uint32_t bp[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = g + ((i >> 1) << 3);
          x[i] = (tok < nv) ? (s[nt][i] + s2[nt][i]) * a.scale_log2 : -INFINITY;
        }
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
        const float corr0 = ex2(m[nt][0] - mn0), corr1 = ex2(m[nt][1] - mn1);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
        const float p0 = ex2(x[0] - mn0), p1 = ex2(x[1] - mn1);
        const float p2 = ex2(x[2] - mn0), p3 = ex2(x[3] - mn1);
        l[nt][0] = l[nt][0] * corr0 + p0 + p2;
        l[nt][1] = l[nt][1] * corr1 + p1 + p3;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][nt][0] *= corr0;
          o[mt][nt][1] *= corr1;
          o[mt][nt][2] *= corr0;
          o[mt][nt][3] *= corr1;
        }
        bp[nt][0] = movmatrix_t(pack_bf16x2(p0, p1));
        bp[nt][1] = movmatrix_t(pack_bf16x2(p2, p3));
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a0, a1, a2, a3;
        uint32_t addr;
        if (TMA) {
          const int cc = 2 * (mt & 3) + (mi & 1);
          addr = vb + (mt >> 2) * half_stride + v_lane_off + ((cc ^ (vt & 7)) << 4);
        } else {
          addr = vb + v_lane_off + mt * 32;
        }
        ldsm_x4_t(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, bp[nt][0], bp[nt][1]);
      }
    }
    if (nv > 0 && nv < 16) fence_proxy_async_smem();  // zeros above, before the next async fill
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    if (h.flags & kSegLast) {
      if (W > 1) {
        // combine the W warps that split this head's tokens (all consumer warps reach the
        // segment end on the same stage)
        float* buf = mbuf + ((size_t)((si > 0 ? si - 1 : 0) * HC + hl) * MF) * 32 + lane;
        if (si > 0) {
          int e = 0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            buf[(e++) * 32] = m[nt][0];
            buf[(e++) * 32] = m[nt][1];
            buf[(e++) * 32] = l[nt][0];
            buf[(e++) * 32] = l[nt][1];
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
              for (int i = 0; i < 4; ++i) buf[(e++) * 32] = o[mt][nt][i];
          }
        }
        named_bar_sync(1, NC * 32);
        if (si == 0) {
          for (int w = 1; w < W; ++w) {
            const float* ob = mbuf + ((size_t)((w - 1) * HC + hl) * MF) * 32 + lane;
            int e = 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float mw0 = ob[(e++) * 32], mw1 = ob[(e++) * 32];
              const float lw0 = ob[(e++) * 32], lw1 = ob[(e++) * 32];
              const float mt0 = fmaxf(m[nt][0], mw0), mt1 = fmaxf(m[nt][1], mw1);
              const float fa0 = ex2(m[nt][0] - mt0), fa1 = ex2(m[nt][1] - mt1);
              const float fb0 = ex2(mw0 - mt0), fb1 = ex2(mw1 - mt1);
              m[nt][0] = mt0;
              m[nt][1] = mt1;
              l[nt][0] = l[nt][0] * fa0 + lw0 * fb0;
              l[nt][1] = l[nt][1] * fa1 + lw1 * fb1;
#pragma unroll
              for (int mt = 0; mt < KS; ++mt) {
                o[mt][nt][0] = o[mt][nt][0] * fa0 + ob[(e++) * 32] * fb0;
                o[mt][nt][1] = o[mt][nt][1] * fa1 + ob[(e++) * 32] * fb1;
                o[mt][nt][2] = o[mt][nt][2] * fa0 + ob[(e++) * 32] * fb0;
                o[mt][nt][3] = o[mt][nt][3] * fa1 + ob[(e++) * 32] * fb1;
              }
            }
          }
        }
        named_bar_sync(1, NC * 32);
      }
      if (si == 0) {
        const bool whole = (h.flags & kStartsUnit) && (h.flags & kEndsUnit);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float lt = l[nt][j];
            lt += __shfl_xor_sync(0xffffffffu, lt, 4);
            lt += __shfl_xor_sync(0xffffffffu, lt, 8);
            lt += __shfl_xor_sync(0xffffffffu, lt, 16);
            const int col = nt * 8 + 2 * c + j;  // query head within the group
            const float inv = 1.f / lt;
            const float lse_v = (m[nt][j] + log2f(lt)) * kLn2;
            if (col < G) {
              const int qhl = hl * G + col;
              if (whole) {
                const int64_t qh = (int64_t)h.hg * HQU + qhl;
                __nv_bfloat16* op = a.out + ((int64_t)h.b * a.num_q_heads + qh) * D;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                  op[mt * 16 + g] = __float2bfloat16_rn(o[mt][nt][j] * inv);
                  op[mt * 16 + g + 8] = __float2bfloat16_rn(o[mt][nt][2 + j] * inv);
                }
                if (g == 0 && a.lse) a.lse[(int64_t)h.b * a.num_q_heads + qh] = lse_v;
              } else {
                float* pp = a.part_o + ((int64_t)h.part * HQU + qhl) * D;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                  pp[mt * 16 + g] = o[mt][nt][j] * inv;
                  pp[mt * 16 + g + 8] = o[mt][nt][2 + j] * inv;
                }
                if (g == 0) a.part_lse[(int64_t)h.part * HQU + qhl] = lse_v;
              }
            }
          }
        }
        if (warp == 0 && lane == 0) {
          if (h.flags & kStartsUnit) a.unit_first[h.unit] = h.part;
          if (h.flags & kEndsUnit) a.unit_last[h.unit] = h.part;
        }
      }
    }
    if (++stage == NS) {
      stage = 0;
      phase ^= 1;
    }
  }
}

template <int D, int NT, bool TMA>
__global__ void __launch_bounds__(288, 1) paged_decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int NS = a.num_stages;
  const int NC = a.HC * a.W;
  if (TMA && (smem_u32(smem) & 1023u)) {  // the swizzled stage layout needs a 1024-byte base
    if (threadIdx.x == 0) report(a.err_word, PKV_DEVERR_INTERNAL);
    return;
  }
  uint8_t* stages = smem;
  const size_t stage_region = (size_t)NS * 2 * a.kv_region;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem + stage_region);
  uint64_t* full = reinterpret_cast<uint64_t*>(hdr + NS);
  uint64_t* empty = full + NS;
  float* mbuf = reinterpret_cast<float*>(empty + NS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    fence_mbar_init();
    if (TMA) {
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  if (warp == NC) {
    decode_producer<D, TMA>(a, stages, hdr, full, empty);
  } else if (warp < NC) {
    decode_consumer<D, NT, TMA>(a, stages, hdr, full, empty, mbuf);
  }
  // Only now may the merge kernel be scheduled (it waits for this grid's completion before
  // reading).  Triggered at the start, its CTAs would sit in their wait for the whole decode and
  // hold the thread slots that kernels on other streams (an extend beside the decode) need on
  // the SMs this grid does not use or has finished with.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// Merge of the decode's split partials: one warp per (unit, query head).  Launched as a
// programmatic dependent of the decode kernel, so it is resident before the decode ends and
// starts as soon as the decode's writes are visible.
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int u = blockIdx.x;
  const int b = u / a.nhg, hg = u % a.nhg;
  const int HQU = a.HC * a.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qhl = blockIdx.y * 8 + warp;
  if (qhl >= HQU) return;
  constexpr int VPL = D / 32;  // values per lane
  const int64_t qh = (int64_t)hg * HQU + qhl;
  const int L = __ldg(a.kv_lens + b);
  if (L <= 0) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(a.err_word, PKV_DEVERR_LENGTH);
    __nv_bfloat16* op = a.out + ((int64_t)b * a.num_q_heads + qh) * D;
#pragma unroll
    for (int i = 0; i < VPL; ++i) op[lane * VPL + i] = __float2bfloat16_rn(0.f);
    if (lane == 0 && a.lse) a.lse[(int64_t)b * a.num_q_heads + qh] = -INFINITY;
    return;
  }
  const int first = a.unit_first[u], last = a.unit_last[u];
  if (first == last) return;  // the decode kernel wrote this unit's output directly
  if (first < 0 || last >= a.num_parts || last < first) {
    if (lane == 0) report(a.err_word, PKV_DEVERR_TIMEOUT);
    return;
  }
  // Every load below is independent of the others in its group, so the merge costs a few L2 round
  // trips whatever the number of partials: the max over all partials' LSE (256 per group), then
  // their weights (read-only-cache hits) and 16 partial rows per lane in flight.
  const float* plse = a.part_lse + qhl;
  float mx = -INFINITY;
  for (int base = first; base <= last; base += 256) {
    float lv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int p = base + 32 * c + lane;
      lv[c] = p <= last ? __ldg(plse + (int64_t)p * HQU) : -INFINITY;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) mx = fmaxf(mx, lv[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  using VecT = typename std::conditional<VPL == 4, float4, float2>::type;
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  float tot = 0.f;
  const float* po = a.part_o + (int64_t)qhl * D + lane * VPL;
  for (int base = first; base <= last; base += 32) {
    const int n = min(32, last - base + 1);
    const float w = lane < n ? __expf(__ldg(plse + (int64_t)(base + lane) * HQU) - mx) : 0.f;
    tot += w;
    for (int i0 = 0; i0 < n; i0 += 16) {
      VecT x[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        x[k] = i0 + k < n ? __ldg(reinterpret_cast<const VecT*>(po + (int64_t)(base + i0 + k) * HQU * D))
                          : VecT{};
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, (i0 + k) & 31);
        const float* xv = reinterpret_cast<const float*>(&x[k]);
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[v] += wk * xv[v];
      }
    }
  }
  tot = warp_sum(tot);
  const float inv = 1.f / tot;
  __nv_bfloat16* op = a.out + ((int64_t)b * a.num_q_heads + qh) * D + lane * VPL;
  if constexpr (VPL == 4) {
    *reinterpret_cast<uint2*>(op) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                               pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(op) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && a.lse) a.lse[(int64_t)b * a.num_q_heads + qh] = mx + logf(tot);
}

// ---------------------------------------------------------------------------------------------
// Generic merge_states: one warp per (row, head); partial states in fp32 or bf16.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__global__ void __launch_bounds__(256) merge_states_kernel(const T* __restrict__ o_parts,
                                                           const float* __restrict__ lse_parts,
                                                           int32_t S, int64_t rows_heads, int32_t D,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int64_t rh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rh >= rows_heads) return;
  // lane i holds the LSEs of splits i, i + 32, ...: the max and the sum are warp reductions
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, __ldg(lse_parts + (int64_t)s * rows_heads + rh));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* op = out + rh * D;
  if (mx == -INFINITY) {  // every split empty
    for (int d = lane * 4; d < D; d += 128)
#pragma unroll
      for (int i = 0; i < 4; ++i) op[d + i] = __float2bfloat16_rn(0.f);
    if (lane == 0 && lse) lse[rh] = -INFINITY;
    return;
  }
  float tot = 0.f;
  // every lane runs every iteration (the shuffles need the whole warp); lanes past D only load
  // and store nothing
  for (int d0 = 0; d0 < D; d0 += 128) {
    const int d = d0 + lane * 4;
    const bool has = d < D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float part = 0.f;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int n = min(32, S - s0);
      // this lane's split weight, shared with the warp by shuffles
      const float wl = lane < n ? __expf(__ldg(lse_parts + (int64_t)(s0 + lane) * rows_heads + rh) - mx) : 0.f;
      part += wl;
      for (int i = 0; i < n; i += 4) {
        float4 v[4];
        float w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // four splits' loads in flight
          w[k] = __shfl_sync(0xffffffffu, wl, (i + k) & 31);
          v[k] = has && i + k < n ? load4(o_parts + ((int64_t)(s0 + i + k) * rows_heads + rh) * D + d)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (i + k < n && w[k] != 0.f) {  // an empty split adds nothing, whatever its o holds
            acc.x += w[k] * v[k].x;
            acc.y += w[k] * v[k].y;
            acc.z += w[k] * v[k].z;
            acc.w += w[k] * v[k].w;
          }
        }
      }
    }
    tot = part;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (has) {
      const float inv = 1.f / tot;
      op[d + 0] = __float2bfloat16_rn(acc.x * inv);
      op[d + 1] = __float2bfloat16_rn(acc.y * inv);
      op[d + 2] = __float2bfloat16_rn(acc.z * inv);
      op[d + 3] = __float2bfloat16_rn(acc.w * inv);
    }
  }
  if (lane == 0 && lse) lse[rh] = mx + logf(tot);
}

// ---------------------------------------------------------------------------------------------
// Host-side planning
// ---------------------------------------------------------------------------------------------
struct DecodePlan {
  int HC, nhg, W, G, NT, Ts, RS, NS;
  bool tma;
  uint32_t region;
  size_t smem;
  int ncta;
  int64_t nunits, nparts;
  size_t off_first, off_last, off_plse, off_po, ws_bytes;
};

constexpr size_t kSmemBudget = 225 * 1024;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool make_plan(int B, int Hq, int Hkv, int D, int ncta, DecodePlan& p, int page_size = 0,
               int64_t num_pages = 0) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return false;
  if (D != 64 && D != 128) return false;
  p.G = Hq / Hkv;
  if (p.G > 16) return false;
  p.NT = (p.G + 7) / 8;
  p.HC = 1;
  for (int d = 1; d <= 8; ++d)
    if (Hkv % d == 0) p.HC = d;
  p.nhg = Hkv / p.HC;
  p.W = 8 / p.HC;
  if (p.W < 1) p.W = 1;
  p.Ts = 16 * p.W;
  const int RB = p.HC * D * 2;
  p.RS = RB + (((RB / 16) % 2 == 0) ? 16 : 0);
  // 16-token slices lie inside one page when the page size is a multiple of 16
  p.tma = page_size > 0 && page_size % 16 == 0 && num_pages * (int64_t)page_size < 0x7fffffffLL;
  p.region = p.tma ? (uint32_t)(D / 64) * p.W * p.HC * 2048 : (uint32_t)(p.Ts * p.RS);
  const size_t stage = (size_t)2 * p.region;
  const int mf = 4 * p.NT + (D / 16) * p.NT * 4;
  const size_t mbytes = p.W > 1 ? (size_t)(p.W - 1) * p.HC * mf * 32 * 4 : 0;
  const size_t fixed = mbytes + (size_t)kMaxStages * (sizeof(StageHdr) + 16);
  if (fixed + 2 * stage > kSmemBudget) return false;
  p.NS = (int)((kSmemBudget - fixed) / stage);
  if (p.NS > kMaxStages) p.NS = kMaxStages;
  p.smem = (size_t)p.NS * stage + (size_t)p.NS * (sizeof(StageHdr) + 16) + mbytes;
  p.ncta = ncta;
  p.nunits = (int64_t)B * p.nhg;
  p.nparts = p.ncta + p.nunits;
  const int HQU = p.HC * p.G;
  p.off_first = 0;
  p.off_last = align256(p.off_first + (size_t)p.nunits * 4);
  p.off_plse = align256(p.off_last + (size_t)p.nunits * 4);
  p.off_po = align256(p.off_plse + (size_t)p.nparts * HQU * 4);
  p.ws_bytes = align256(p.off_po + (size_t)p.nparts * HQU * D * 4);
  return true;
}

template <int D, int NT, bool TMA>
pkv_status launch_decode(const DecodePlan& p, const DecodeArgs& a, cudaStream_t st) {
  auto kern = paged_decode_kernel<D, NT, TMA>;
  // the dynamic shared-memory limit this instance was raised to, per device (any host thread)
  static std::atomic<int> configured_dev[64];
  const int dev = pkv_host::current_device();
  if (dev < 0) return PKV_ERR_CUDA;
  if (dev >= 64 || configured_dev[dev].load(std::memory_order_relaxed) < (int)p.smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) {
      int cur = configured_dev[dev].load(std::memory_order_relaxed);
      while (cur < (int)p.smem &&
             !configured_dev[dev].compare_exchange_weak(cur, (int)p.smem, std::memory_order_relaxed)) {
      }
    }
  }
  const int threads = (p.HC * p.W + 1) * 32;
  kern<<<p.ncta, threads, p.smem, st>>>(a);
  pkv_status s = pkv_host::launch_status();
  if (s != PKV_OK) return s;
  if (p.nunits > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nunits, (unsigned)((p.HC * p.G + 7) / 8), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, a) != cudaSuccess) return PKV_ERR_CUDA;
    s = pkv_host::launch_status();
  }
  return s;
}

}  // namespace

extern "C" {

size_t pkv_decode_workspace_size(int32_t batch_size, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim) {
  DecodePlan p;
  const int n = pkv_host::sm_count();
  if (n <= 0) return 0;
  if (!make_plan(batch_size, num_q_heads, num_kv_heads, head_dim, n, p)) return 0;
  return p.ws_bytes;
}

pkv_status pkv_paged_decode(const pkv_pool* pool, const void* q, int32_t batch_size,
                            int32_t num_q_heads, const int32_t* kv_indptr,
                            const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            uint32_t* err_word, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_decode");
  return pkv_paged_decode_ctas(pool, q, batch_size, num_q_heads, kv_indptr, kv_indices, kv_lens,
                               sm_scale, out, lse, workspace, workspace_bytes, err_word, 0, stream);
}

pkv_status pkv_paged_decode_ctas(const pkv_pool* pool, const void* q, int32_t batch_size,
                                 int32_t num_q_heads, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 uint32_t* err_word, int32_t max_ctas, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_decode_ctas");
  return pkv_paged_decode_l2keep(pool, q, batch_size, num_q_heads, kv_indptr, kv_indices, kv_lens, sm_scale,
                                 out, lse, workspace, workspace_bytes, err_word, max_ctas, nullptr, stream);
}

pkv_status pkv_paged_decode_l2keep(const pkv_pool* pool, const void* q, int32_t batch_size,
                                   int32_t num_q_heads, const int32_t* kv_indptr,
                                   const int32_t* kv_indices, const int32_t* kv_lens, float sm_scale,
                                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                                   uint32_t* err_word, int32_t max_ctas, const int32_t* keep_tokens,
                                   void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_decode_l2keep");
  if (!pkv_host::valid_pool(pool) || batch_size < 0 || num_q_heads <= 0 || max_ctas < 0)
    return PKV_ERR_INVALID_ARG;
  if (batch_size == 0) return PKV_OK;
  if (!q || !kv_indptr || !kv_indices || !kv_lens || !out) return PKV_ERR_INVALID_ARG;
  if (!pkv_host::aligned16(q) || !pkv_host::aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (batch_size > 0x7fffffff / 64) return PKV_ERR_UNSUPPORTED;
  const int D = pool->head_dim;
  int ncta = pkv_host::sm_count();
  if (ncta <= 0) return PKV_ERR_CUDA;
  if (max_ctas > 0 && max_ctas < ncta) ncta = max_ctas;  // fewer partials: the workspace still fits
  DecodePlan p;
  if (!make_plan(batch_size, num_q_heads, pool->num_kv_heads, D, ncta, p, pool->page_size, pool->num_pages))
    return PKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < p.ws_bytes) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_INVALID_ARG;

  DecodeArgs a;
  a.k_pool = (const __nv_bfloat16*)pool->k;
  a.v_pool = (const __nv_bfloat16*)pool->v;
  a.num_pages = pool->num_pages;
  a.page_size = pool->page_size;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = (const __nv_bfloat16*)q;
  a.batch = batch_size;
  a.num_q_heads = num_q_heads;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.kv_lens = kv_lens;
  a.keep_tokens = keep_tokens;
  a.scale_log2 = sm_scale * pkv::kLog2e;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  uint8_t* ws = (uint8_t*)workspace;
  a.unit_first = (int32_t*)(ws + p.off_first);
  a.unit_last = (int32_t*)(ws + p.off_last);
  a.part_lse = (float*)(ws + p.off_plse);
  a.part_o = (float*)(ws + p.off_po);
  a.err_word = err_word;
  a.HC = p.HC;
  a.nhg = p.nhg;
  a.W = p.W;
  a.group = p.G;
  a.row_stride = p.RS;
  a.stage_tokens = p.Ts;
  a.num_stages = p.NS;
  a.num_parts = (int32_t)p.nparts;
  a.kv_region = p.region;
  bool tma = p.tma;
  if (tma) {
    const uint64_t Hkv = pool->num_kv_heads;
    const uint64_t rows = (uint64_t)pool->num_pages * pool->page_size;
    tma = pkv_host::encode_tmap_3d(&a.tm_k, pool->k, D, rows, Hkv, Hkv * D * 2, (uint64_t)D * 2, 64, 16,
                                   p.HC) &&
          pkv_host::encode_tmap_3d(&a.tm_v, pool->v, D, rows, Hkv, Hkv * D * 2, (uint64_t)D * 2, 64, 16,
                                   p.HC);
    if (!tma) {  // fall back to row copies with the matching stage layout
      p.tma = false;
      if (!make_plan(batch_size, num_q_heads, pool->num_kv_heads, D, ncta, p)) return PKV_ERR_UNSUPPORTED;
      a.num_stages = p.NS;
      a.kv_region = p.region;
    }
  }

  cudaStream_t st = (cudaStream_t)stream;
  if (p.tma) {
    if (D == 128) return p.NT == 1 ? launch_decode<128, 1, true>(p, a, st) : launch_decode<128, 2, true>(p, a, st);
    return p.NT == 1 ? launch_decode<64, 1, true>(p, a, st) : launch_decode<64, 2, true>(p, a, st);
  }
  if (D == 128) return p.NT == 1 ? launch_decode<128, 1, false>(p, a, st) : launch_decode<128, 2, false>(p, a, st);
  return p.NT == 1 ? launch_decode<64, 1, false>(p, a, st) : launch_decode<64, 2, false>(p, a, st);
}

}  // extern "C"

namespace {

template <typename T>
pkv_status launch_merge_states(const T* o_parts, const float* lse_parts, int32_t num_splits,
                               int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                               float* lse, void* stream) {
  if (num_splits < 0 || num_rows < 0 || num_heads <= 0 || head_dim <= 0) return PKV_ERR_INVALID_ARG;
  if (num_rows == 0) return PKV_OK;
  if (!o_parts || !lse_parts || !out || num_splits == 0) return PKV_ERR_INVALID_ARG;
  if (head_dim % 4 != 0 || head_dim > 512) return PKV_ERR_UNSUPPORTED;
  if (!pkv_host::aligned16(o_parts)) return PKV_ERR_INVALID_ARG;
  const int64_t rh = (int64_t)num_rows * num_heads;
  const int warps = 8;
  const int64_t blocks = (rh + warps - 1) / warps;
  if (blocks > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
  merge_states_kernel<T><<<(unsigned)blocks, warps * 32, 0, (cudaStream_t)stream>>>(
      o_parts, lse_parts, num_splits, rh, head_dim, (__nv_bfloat16*)out, lse);
  return pkv_host::launch_status();
}

}  // namespace

extern "C" {

pkv_status pkv_merge_states(const float* o_parts, const float* lse_parts, int32_t num_splits,
                            int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                            float* lse, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_merge_states");
  return launch_merge_states(o_parts, lse_parts, num_splits, num_rows, num_heads, head_dim, out, lse,
                             stream);
}

pkv_status pkv_merge_states_bf16(const void* o_parts, const float* lse_parts, int32_t num_splits,
                                 int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                                 float* lse, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_merge_states_bf16");
  return launch_merge_states((const __nv_bfloat16*)o_parts, lse_parts, num_splits, num_rows, num_heads,
                             head_dim, out, lse, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Decode without a caller-supplied workspace.
//
// Some callers cannot allocate device memory when they need a decode: a serving engine that
// reserves a fixed share of HBM for its KV pool up front leaves nothing for per-call buffers,
// and code that must not take cudaMalloc's implicit device-wide synchronisation (or its failure
// modes) in the middle of a step has no safe place to get a workspace either.  For them the
// split partials live in one file-scope device array, sized once, held by every GPU that loads
// this library for as long as the process lives.
// ---------------------------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_decode_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};
unsigned long long g_scratch_ctx[64] = {0};  // context the cached address belongs to

// Device address of g_decode_scratch on the current device (in host code the array's name is
// only a stand-in for the symbol, never a device pointer).  Looked up once per device, and again
// when the device's context has changed (after a cudaDeviceReset the old address is gone).
void* scratch_on_current_device() {
  const int dev = pkv_host::current_device();
  if (dev < 0 || dev >= 64) return nullptr;
  const unsigned long long ctx = pkv_host::current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
    // the lookup creates the context if there was none yet
    g_scratch_ctx[dev] = ctx != 0 ? ctx : pkv_host::current_context_id();
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_noalloc(const pkv_pool* pool, const void* q, int32_t batch_size,
                                               int32_t num_q_heads, const int32_t* kv_indptr,
                                               const int32_t* kv_indices, const int32_t* kv_lens,
                                               float sm_scale, void* out, float* lse,
                                               uint32_t* err_word, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_paged_decode_noalloc");
  if (!pkv_host::valid_pool(pool) || batch_size < 0 || num_q_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (batch_size == 0) return PKV_OK;
  const int n = pkv_host::sm_count();
  if (n <= 0) return PKV_ERR_CUDA;
  DecodePlan p;
  if (!make_plan(batch_size, num_q_heads, pool->num_kv_heads, pool->head_dim, n, p)) {
    // let the regular entry point classify the shape error
    return pkv_paged_decode(pool, q, batch_size, num_q_heads, kv_indptr, kv_indices, kv_lens,
                            sm_scale, out, lse, nullptr, 0, err_word, stream);
  }
  if (p.ws_bytes > (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return PKV_ERR_CUDA;
  // The partials need no initial contents: every slot a merge reads is written earlier in the
  // same call.  Calls that overlap on the GPU (other streams) share the array and race.
  return pkv_paged_decode(pool, q, batch_size, num_q_heads, kv_indptr, kv_indices, kv_lens, sm_scale,
                          out, lse, ws, (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES, err_word, stream);
}
