// KV-cache write fused with the rotary position embedding of the step's new K (and, optionally,
// its Q): the step just before attention in the engines' forward pass, done in the same pass that
// writes K/V into the pool so K is read and written once.
//
// Rotation: half-split pairing (the rotate_half convention of HF Llama/Qwen checkpoints that the
// nanoSGLang README, "Notable Fixes", settles on): for i < D/2,
//   x'[i] = x[i] cos(a_i) - x[i + D/2] sin(a_i),  x'[i + D/2] = x[i + D/2] cos(a_i) + x[i] sin(a_i),
// a_i = position * theta^(-2i/D), with cos and sin read from a caller-provided fp32 table.
// HBM-bound: one thread per 8 pairs (16 bytes of each half) of one head of one token.
#include "common.cuh"

namespace {

using namespace pkv;

PKV_DEV void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

PKV_DEV uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

PKV_DEV void rotate8(const float (&lo)[8], const float (&hi)[8], const float4 c0, const float4 c1,
                     const float4 s0, const float4 s1, float (&olo)[8], float (&ohi)[8]) {
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    olo[i] = fmaf(lo[i], c[i], -hi[i] * s[i]);
    ohi[i] = fmaf(hi[i], c[i], lo[i] * s[i]);
  }
}

__global__ void __launch_bounds__(256) rope_append_kernel(
    __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool,
    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
    __nv_bfloat16* __restrict__ q, const int64_t* __restrict__ slots, const int32_t* __restrict__ positions,
    const float* __restrict__ cos_sin, int32_t max_position, int32_t T, int32_t Hkv, int32_t Hq_rot,
    int32_t D, int64_t num_slots, uint32_t* err_word) {
  const int chunks = D / 16;  // 8-pair chunks per head
  const int heads = Hkv + Hq_rot;
  const int64_t total = (int64_t)T * heads * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % chunks);
    const int64_t th = i / chunks;
    const int h = (int)(th % heads);
    const int64_t t = th / heads;
    const int32_t pos = __ldg(positions + t);
    if (pos < 0 || pos >= max_position) {
      if (h == 0 && c == 0) report(err_word, PKV_DEVERR_LENGTH);
      continue;
    }
    const float4* cs = reinterpret_cast<const float4*>(cos_sin + (int64_t)pos * D);
    const float4 c0 = __ldg(cs + 2 * c), c1 = __ldg(cs + 2 * c + 1);
    const float4 s0 = __ldg(cs + D / 8 + 2 * c), s1 = __ldg(cs + D / 8 + 2 * c + 1);
    float lo[8], hi[8], olo[8], ohi[8];
    if (h < Hkv) {
      const int64_t slot = __ldg(slots + t);
      if (slot < 0) continue;  // padding token
      if (slot >= num_slots) {
        if (c == 0) report(err_word, PKV_DEVERR_SLOT_OOB);
        continue;
      }
      const int64_t src = (t * Hkv + h) * D + 8 * c;
      const int64_t dst = (slot * Hkv + h) * D + 8 * c;
      unpack8(__ldg(reinterpret_cast<const uint4*>(k_new + src)), lo);
      unpack8(__ldg(reinterpret_cast<const uint4*>(k_new + src + D / 2)), hi);
      rotate8(lo, hi, c0, c1, s0, s1, olo, ohi);
      *reinterpret_cast<uint4*>(k_pool + dst) = pack8(olo);
      *reinterpret_cast<uint4*>(k_pool + dst + D / 2) = pack8(ohi);
      *reinterpret_cast<uint4*>(v_pool + dst) = __ldg(reinterpret_cast<const uint4*>(v_new + src));
      *reinterpret_cast<uint4*>(v_pool + dst + D / 2) = __ldg(reinterpret_cast<const uint4*>(v_new + src + D / 2));
    } else {
      __nv_bfloat16* x = q + (t * Hq_rot + (h - Hkv)) * D + 8 * c;
      unpack8(*reinterpret_cast<const uint4*>(x), lo);
      unpack8(*reinterpret_cast<const uint4*>(x + D / 2), hi);
      rotate8(lo, hi, c0, c1, s0, s1, olo, ohi);
      *reinterpret_cast<uint4*>(x) = pack8(olo);
      *reinterpret_cast<uint4*>(x + D / 2) = pack8(ohi);
    }
  }
}

}  // namespace

extern "C" pkv_status pkv_rope_kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                                         const int64_t* slot_mapping, const int32_t* positions,
                                         const float* cos_sin, int32_t max_position, void* q,
                                         int32_t num_q_heads, int32_t num_tokens, uint32_t* err_word,
                                         void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_rope_kv_append");
  if (!pkv_host::valid_pool(pool) || num_tokens < 0 || num_q_heads < 0 || max_position <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !positions || !cos_sin) return PKV_ERR_INVALID_ARG;
  if (q == nullptr && num_q_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!pkv_host::aligned16(k_new) || !pkv_host::aligned16(v_new) || !pkv_host::aligned16(cos_sin) ||
      (q && !pkv_host::aligned16(q)))
    return PKV_ERR_INVALID_ARG;
  if (pool->head_dim % 16 != 0) return PKV_ERR_UNSUPPORTED;
  const int heads = pool->num_kv_heads + (q ? num_q_heads : 0);
  const int64_t total = (int64_t)num_tokens * heads * (pool->head_dim / 16);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)pkv_host::sm_count() * 16;
  if (cap > 0 && blocks > cap) blocks = cap;
  rope_append_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      (__nv_bfloat16*)pool->k, (__nv_bfloat16*)pool->v, (const __nv_bfloat16*)k_new,
      (const __nv_bfloat16*)v_new, (__nv_bfloat16*)q, slot_mapping, positions, cos_sin, max_position,
      num_tokens, pool->num_kv_heads, q ? num_q_heads : 0, pool->head_dim,
      pool->num_pages * pool->page_size, err_word);
  return pkv_host::launch_status();
}

// ---------------------------------------------------------------------------------------------
// The cos/sin table the fused append reads.  Row p, column i < D/2: cos(a), column D/2 + i:
// sin(a), with the angle a = p * theta^(-2i/D) of pair i at position p (the half-split rotary
// embedding of HF Llama/Qwen checkpoints, nanoSGLang README "Notable Fixes").  The angle is
// formed in double precision, so that large positions keep it to well under an fp32 ulp of the
// cosine, and cos/sin come from CUDA's double-precision sincos before the fp32 rounding.  Built
// once, like a model's rotary buffer; the double-precision work (~2M angles for 32K positions of
// D = 128) takes well under a millisecond.
// ---------------------------------------------------------------------------------------------
namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(float* __restrict__ table, int32_t max_position,
                                                        int32_t head_dim, double theta) {
  const int half = head_dim / 2;
  const int64_t n = (int64_t)max_position * half;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = idx / half;
    const int i = (int)(idx - p * half);
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    table[p * head_dim + i] = (float)c;
    table[p * head_dim + half + i] = (float)s;
  }
}

}  // namespace

extern "C" pkv_status pkv_rope_cos_sin_table(float* table, int32_t max_position, int32_t head_dim,
                                             double theta, void* stream) {
  pkv_host::NvtxRange nvtx_range("pkv_rope_cos_sin_table");
  if (max_position < 0 || head_dim <= 0 || head_dim % 2 != 0 || !(theta > 0.0)) return PKV_ERR_INVALID_ARG;
  if (max_position == 0) return PKV_OK;
  if (!table) return PKV_ERR_INVALID_ARG;
  const int64_t n = (int64_t)max_position * (head_dim / 2);
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  const int64_t cap = (int64_t)pkv_host::sm_count() * 8;
  if (cap > 0 && blocks > cap) blocks = cap;
  rope_table_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(table, max_position, head_dim,
                                                                            theta);
  return pkv_host::launch_status();
}
