// Decode attention on the paged TurboQuant cache (libtq, sm_103a).
//
// What is computed (issoh.co.jp TurboQuant overview, §第1段/§第2段; lilting.ch
// TurboQuant article, QJL section; bf16 boundary layers per the overview's
// §起動コマンド):
//   q' = Pi q once per query head (scaled by sm_scale * log2 e),
//   u_t = gamma_t <q', c_K[idx_t]> (+ sqrt(pi/2)/m rho_t <S q', 2 sigma_t - 1>),
//   online softmax over the context in base 2, value accumulation in the
//   rotated domain  acc = sum_t 2^(u_t - M) gamma'_t c_V[idx'_t],
//   and o = Pi^T (acc / l) once per query head.  Dequantized K/V never reach HBM.
//
// Kernels and launch shapes:
//   k_rotate_q     warp per (sequence, query head): FWHT or dense mat-vec.
//   k_decode_*     CTA per (split, kv head [, head group], sequence), 4 warps.
//                  Each warp streams its own blocks of the split: the K and V
//                  pages of a block are brought into shared memory by two 1-D
//                  bulk copies (cp.async.bulk, completion on an mbarrier) in a
//                  4-deep ring.  Codes are decoded to fp16 centroids in
//                  registers (prmt lookups on 8-entry tables) straight into
//                  mma.sync m16n8k16 fragments: logits^T = Q'(16 rows = 8 heads
//                  x {hi, lo} fp16 split) x K_hat^T, then acc^T += V_hat^T x P'^T
//                  where P'_t = 2^(u_t - M) gamma'_t / W_block (<= 1 in fp16) and
//                  W_block is folded back in fp32.
//   k_combine      CTA per (sequence, query head): log-sum-exp merge of the
//                  splits and the inverse rotation.
#include <cfloat>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kWarps = 4;
constexpr int kStages = 4;
constexpr float kRescaleThreshold = 20.0f;  // log2 units before the running max is refreshed
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after ~1 s (returns false).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63) == 63 && global_ns() - t0 > 1000000000ull) return false;
  }
  return false;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                        const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------- code -> fp16 decode

// fp16 centroid table split into byte planes for prmt lookups.
// BITS == 4: the 8 positive magnitudes c[8 + m] (the sign comes from the code);
// BITS <= 3: the 2^BITS signed centroids c[e] directly.
struct HalfTable {
  uint32_t lo0, lo1, hi0, hi1;
};

template <int BITS>
__device__ __forceinline__ HalfTable make_table(const Codebook& cb) {
  uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float v = 0.0f;
    if (BITS == 4) v = cb.c[8 + e];
    else if (e < (1 << BITS)) v = cb.c[e];
    const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(v));
    lo[e >> 2] |= (h & 0xFFu) << (8 * (e & 3));
    hi[e >> 2] |= (h >> 8) << (8 * (e & 3));
  }
  return HalfTable{lo[0], lo[1], hi[0], hi[1]};
}

// Looks up 4 codes held in the 4 nibbles of `nib` (bits 0..15).  Returns the
// low bytes and high bytes of the 4 fp16 centroids (byte k <-> nibble k).
template <int BITS>
__device__ __forceinline__ void lookup4(uint32_t nib, const HalfTable& t, uint32_t& lo, uint32_t& hi) {
  if constexpr (BITS == 4) {
    // codes 0..7 are the negatives of magnitude 7 - code, codes 8..15 magnitude code - 8
    const uint32_t neg = ~nib & 0x8888u;
    const uint32_t sel = (nib ^ (neg - (neg >> 3))) & 0x7777u;
    lo = prmt(t.lo0, t.lo1, sel);
    hi = prmt(t.hi0, t.hi1, sel);
    // sign byte k = replicated flag of nibble k (flags at bit 7 of (neg << 4) / neg bytes)
    const uint32_t sgn = prmt(neg << 4, neg, 0xD9C8u);
    hi ^= sgn & 0x80808080u;
  } else {
    lo = prmt(t.lo0, t.lo1, nib);
    hi = prmt(t.hi0, t.hi1, nib);
  }
}

// 3-bit codes of a 24-bit group -> one code per nibble.
__device__ __forceinline__ uint32_t spread3(uint32_t x) {
  uint32_t t = (x & 0xFFFu) | ((x & 0xFFF000u) << 4);
  t = (t & 0x003F003Fu) | ((t & 0x0FC00FC0u) << 2);
  return (t & 0x07070707u) | ((t & 0x38383838u) << 1);
}

// 2-bit codes of a 16-bit group -> one code per nibble.
__device__ __forceinline__ uint32_t spread2(uint32_t x) {
  uint32_t t = (x & 0xFFu) | ((x & 0xFF00u) << 8);
  t = (t & 0x000F000Fu) | ((t & 0x00F000F0u) << 4);
  return (t & 0x03030303u) | ((t & 0x0C0C0C0Cu) << 2);
}

// The 32 codes of quarter `tig` of a record (coordinates [32 tig, 32 tig + 32))
// as 4 nibble words of 8 codes.
template <int BITS>
__device__ __forceinline__ void load_quarter(const uint8_t* rec, int tig, uint32_t (&nw)[4]) {
  if constexpr (BITS == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(rec + 16 * tig);
    nw[0] = v.x; nw[1] = v.y; nw[2] = v.z; nw[3] = v.w;
  } else if constexpr (BITS == 3) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(rec + 12 * tig);
    const uint32_t w0 = p[0], w1 = p[1], w2 = p[2];
    nw[0] = spread3(w0 & 0xFFFFFFu);
    nw[1] = spread3((w0 >> 24) | ((w1 & 0xFFFFu) << 8));
    nw[2] = spread3((w1 >> 16) | ((w2 & 0xFFu) << 16));
    nw[3] = spread3(w2 >> 8);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(rec + 8 * tig);
    nw[0] = spread2(v.x & 0xFFFFu);
    nw[1] = spread2(v.x >> 16);
    nw[2] = spread2(v.y & 0xFFFFu);
    nw[3] = spread2(v.y >> 16);
  }
}

// The 16 codes of coordinates [16 g, 16 g + 16) of a record as 2 nibble words.
template <int BITS>
__device__ __forceinline__ void load_sixteenth(const uint8_t* rec, int g, uint32_t (&nw)[2]) {
  if constexpr (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(rec + 8 * g);
    nw[0] = v.x; nw[1] = v.y;
  } else if constexpr (BITS == 3) {
    const int byte = 6 * g;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(rec + (byte & ~3));
    const uint64_t z = ((uint64_t)p[1] << 32 | p[0]) >> (8 * (byte & 3));
    nw[0] = spread3((uint32_t)z & 0xFFFFFFu);
    nw[1] = spread3((uint32_t)(z >> 24) & 0xFFFFFFu);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + 4 * g);
    nw[0] = spread2(w & 0xFFFFu);
    nw[1] = spread2(w >> 16);
  }
}

// ------------------------------------------------------------ shared pieces

struct DecodeArgs {
  const uint8_t* kpool;
  const uint8_t* vpool;
  int kpage, vpage;  // bytes per page
  int Hkv;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* ctx_lens;
  const float* qrot;  // [B][Hq][d] scaled rotated queries
  const float* uqjl;  // [B][Hq][d] S q' (QJL only)
  int Hq, g, ngroups;
  int splits;
  float* part;  // [B][Hq][splits][d]
  float* ml;    // [B][Hq][splits][2]
  Codebook cbk, cbv;
  float qjl_coef;  // sqrt(pi/2) / m
  unsigned* status;
};

// Splits one fp32 query row (32 coordinates of quarter tig) into the hi/lo
// fp16 A fragments of 8 k-chunks.  Returns 1/scale.
__device__ __forceinline__ float make_q_frags(const float* qrow, bool valid, int tig, uint32_t (&a)[8][4]) {
  float v[32];
  if (valid) {
    load32<float>(qrow + 32 * tig, v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  }
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
  mx = quad_max(mx);
  int e = 0;
  if (mx > 0.0f) frexpf(mx, &e);
  const float scale = ldexpf(1.0f, 14 - e);  // max |q| * scale < 2^14
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float s = v[4 * c + k] * scale;
      hi[k] = __half2float(__float2half_rn(s));
      lo[k] = s - hi[k];
    }
    a[c][0] = pack_half2(hi[0], hi[1]);
    a[c][1] = pack_half2(lo[0], lo[1]);
    a[c][2] = pack_half2(hi[2], hi[3]);
    a[c][3] = pack_half2(lo[2], lo[3]);
  }
  return 1.0f / scale;
}

// Online-softmax state of one warp: running max M and partial denominator l
// for head g_ (row of the thread), rotated-domain accumulator fragments
// acc[i] = columns (heads 2 tig, 2 tig + 1) x rows (coords 16 g_ + 2i, +1).
struct SoftmaxState {
  float M, l;
  float acc[8][4];
};

// Given the 4 scaled logits u (tokens 2tig, 2tig+1, 8+2tig, 9+2tig) and value
// weights wv (gamma' or 1), updates M, l, rescales acc when needed and returns
// the fp16 B fragments of P' plus the per-column block weights.
__device__ __forceinline__ void softmax_block(SoftmaxState& st, const float (&u)[4], const float (&wv)[4], int lane,
                                              int tig, uint32_t& bp0, uint32_t& bp1, float& W0, float& W1,
                                              bool bf16_p, uint32_t* bp_lo0 = nullptr, uint32_t* bp_lo1 = nullptr) {
  float bmax = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
  bmax = quad_max(bmax);
  const bool need = bmax > st.M + kRescaleThreshold;
  if (__any_sync(0xffffffffu, need)) {
    const float newM = need ? bmax : st.M;
    const float alpha = (st.M == -INFINITY) ? 0.0f : exp2f(st.M - newM);
    st.l *= alpha;
    st.M = newM;
    const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * tig) * 4);
    const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * tig + 1) * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.acc[i][0] *= a0; st.acc[i][1] *= a1; st.acc[i][2] *= a0; st.acc[i][3] *= a1;
    }
  }
  float p[4], w[4];
  float wmax = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    p[e] = exp2f(u[e] - st.M);
    st.l += p[e];
    w[e] = p[e] * wv[e];
    wmax = fmaxf(wmax, w[e]);
  }
  wmax = quad_max(wmax);
  const float rW = wmax > 0.0f ? 1.0f / wmax : 0.0f;
  float pn[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) pn[e] = w[e] * rW;
  if (bf16_p) {
    bp0 = pack_bf162(pn[0], pn[1]);
    bp1 = pack_bf162(pn[2], pn[3]);
    const __nv_bfloat162 h0 = *reinterpret_cast<__nv_bfloat162*>(&bp0);
    const __nv_bfloat162 h1 = *reinterpret_cast<__nv_bfloat162*>(&bp1);
    *bp_lo0 = pack_bf162(pn[0] - __low2float(h0), pn[1] - __high2float(h0));
    *bp_lo1 = pack_bf162(pn[2] - __low2float(h1), pn[3] - __high2float(h1));
  } else {
    bp0 = pack_half2(pn[0], pn[1]);
    bp1 = pack_half2(pn[2], pn[3]);
  }
  W0 = __shfl_sync(0xffffffffu, wmax, (2 * tig) * 4);
  W1 = __shfl_sync(0xffffffffu, wmax, (2 * tig + 1) * 4);
  (void)lane;
}

// Merges the 4 warps' states through shared memory and writes the split's
// partial (acc[d], M, l) for every head of the CTA.
__device__ __forceinline__ void write_partials(SoftmaxState& st, float* red, int warp, int lane, int gc,
                                               const DecodeArgs& a, int b, int head0, int split) {
  const int g_ = lane >> 2, tig = lane & 3;
  st.l = quad_sum(st.l);
  float* racc = red;                        // [4 warps][8 heads][128]
  float* rm = red + kWarps * 8 * kD;        // [4][8]
  float* rl = rm + kWarps * 8;              // [4][8]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c0 = 16 * g_ + 2 * i;
    float* base = racc + warp * 8 * kD;
    base[(2 * tig) * kD + c0] = st.acc[i][0];
    base[(2 * tig + 1) * kD + c0] = st.acc[i][1];
    base[(2 * tig) * kD + c0 + 1] = st.acc[i][2];
    base[(2 * tig + 1) * kD + c0 + 1] = st.acc[i][3];
  }
  if (tig == 0) {
    rm[warp * 8 + g_] = st.M;
    rl[warp * 8 + g_] = st.l;
  }
  __syncthreads();
  const int t = threadIdx.x;  // coordinate
  for (int h = 0; h < gc; ++h) {
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Mt = fmaxf(Mt, rm[w * 8 + h]);
    float acc = 0.0f, L = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = rm[w * 8 + h];
      const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - Mt);
      acc += racc[(w * 8 + h) * kD + t] * f;
      L += rl[w * 8 + h] * f;
    }
    const int64_t row = ((int64_t)b * a.Hq + head0 + h) * a.splits + split;
    a.part[row * kD + t] = acc;
    if (t == 0) {
      a.ml[row * 2] = Mt;
      a.ml[row * 2 + 1] = L;
    }
  }
}

// Per-warp ring of (K page, V page) stages fed by bulk copies.
struct Ring {
  uint8_t* buf;   // kStages x (kpage + vpage)
  uint64_t* bar;  // kStages
  int stage_bytes;
};

// Issues the copies of block j of the sequence into `stage` (lane 0 only).
// Returns true (on every lane) if the block id was valid and copies were issued.
__device__ __forceinline__ bool issue_block(const Ring& r, int stage, const DecodeArgs& a, int b, int kvh, int j,
                                            int lane) {
  int blk = 0;
  if (lane == 0) blk = __ldg(a.block_table + (int64_t)b * a.max_blocks + j);
  blk = __shfl_sync(0xffffffffu, blk, 0);
  const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
  if (lane == 0) {
    uint64_t* bar = r.bar + stage;
    if (ok) {
      uint8_t* dst = r.buf + stage * r.stage_bytes;
      const uint8_t* srck = a.kpool + ((int64_t)blk * a.Hkv + kvh) * a.kpage;
      const uint8_t* srcv = a.vpool + ((int64_t)blk * a.Hkv + kvh) * a.vpage;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(bar, (uint32_t)(a.kpage + a.vpage));
      bulk_copy_g2s(dst, srck, (uint32_t)a.kpage, bar);
      bulk_copy_g2s(dst + a.kpage, srcv, (uint32_t)a.vpage, bar);
    } else {
      flag_status(a.status, TQ_DEV_BAD_BLOCK);
      mbar_arrive(bar);  // completes the phase without data
    }
  }
  return ok;
}

// ----------------------------------------------------- packed decode kernel

template <int BK, int BV, bool QJL>
__global__ void __launch_bounds__(kWarps * 32) k_decode_packed(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int RK = 16 * BK, RV = 16 * BV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_ = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.ngroups, hg = blockIdx.y % a.ngroups;
  const int b = blockIdx.z;
  const int head0 = kvh * a.g + hg * 8;
  const int gc = min(8, a.g - hg * 8);

  int ctx = __ldg(a.ctx_lens + b);
  if (ctx < 0 || ctx > a.max_blocks * kBlock) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_status(a.status, TQ_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : a.max_blocks * kBlock;
  }
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int j0 = (int)((int64_t)split * nblk / a.splits);
  const int j1 = (int)((int64_t)(split + 1) * nblk / a.splits);
  const int n_my = j1 - j0 > warp ? (j1 - j0 - warp + kWarps - 1) / kWarps : 0;

  const int stage_bytes = a.kpage + a.vpage;
  Ring ring;
  ring.stage_bytes = stage_bytes;
  ring.buf = smem_raw + warp * kStages * stage_bytes;
  ring.bar = reinterpret_cast<uint64_t*>(smem_raw + kWarps * kStages * stage_bytes) + warp * kStages;
  if (lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(ring.bar + s, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();

  // prologue copies
  uint32_t valid_mask = 0u;
  for (int s = 0; s < kStages && s < n_my; ++s)
    if (issue_block(ring, s, a, b, kvh, j0 + warp + kWarps * s, lane)) valid_mask |= 1u << s;

  // query fragments (rows g_ < gc hold head head0 + g_)
  uint32_t aq[8][4];
  const bool hv = g_ < gc;
  const float inv_qs = make_q_frags(a.qrot + ((int64_t)b * a.Hq + head0 + (hv ? g_ : 0)) * kD, hv, tig, aq);
  uint32_t au[8][4];
  float inv_us = 0.0f;
  if constexpr (QJL) inv_us = make_q_frags(a.uqjl + ((int64_t)b * a.Hq + head0 + (hv ? g_ : 0)) * kD, hv, tig, au);

  const HalfTable tk = make_table<BK>(a.cbk);
  const HalfTable tv = make_table<BV>(a.cbv);

  SoftmaxState st;
  st.M = -INFINITY;
  st.l = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.acc[i][0] = st.acc[i][1] = st.acc[i][2] = st.acc[i][3] = 0.0f;
  const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};

  int i = 0;
  bool aborted = false;
  for (; i < n_my; ++i) {
    const int stage = i % kStages;
    const uint32_t parity = (uint32_t)(i / kStages) & 1u;
    if (!mbar_wait(ring.bar + stage, parity)) {
      if (lane == 0) flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    const int j = j0 + warp + kWarps * i;
    if (valid_mask & (1u << stage)) {
      const uint8_t* sk = ring.buf + stage * stage_bytes;
      const uint8_t* sv = sk + a.kpage;
      const int t0 = j * kBlock;

      // logits^T = Q' K_hat^T for tokens 0..7 (n-tile 0) and 8..15 (n-tile 1)
      float s[2][4], sq[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint32_t kn[4];
        load_quarter<BK>(sk + (8 * nt + g_) * RK, tig, kn);
        float accs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t nib = (c & 1) ? (kn[c >> 1] >> 16) : (kn[c >> 1] & 0xFFFFu);
          uint32_t lo, hi;
          lookup4<BK>(nib, tk, lo, hi);
          mma_f16(accs, aq[c], prmt(lo, hi, 0x5140u), prmt(lo, hi, 0x7362u), accs);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = accs[e];
        if constexpr (QJL) {
          const uint32_t sw = *reinterpret_cast<const uint32_t*>(sk + 16 * RK + 64 + 16 * (8 * nt + g_) + 4 * tig);
          float accq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t nb = ~(sw >> (4 * c));
            const uint32_t b0 = 0x3C003C00u | ((nb & 1u) << 15) | ((nb & 2u) << 30);
            const uint32_t b1 = 0x3C003C00u | ((nb & 4u) << 13) | ((nb & 8u) << 28);
            mma_f16(accq, au[c], b0, b1, accq);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sq[nt][e] = accq[e];
        }
      }
      // scaled logits of tokens 2tig, 2tig+1 (nt 0) and 8+2tig, 9+2tig (nt 1)
      float u[4], wv[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float2 gk = *reinterpret_cast<const float2*>(sk + 16 * RK + 4 * (8 * nt + 2 * tig));
        const float2 gv = *reinterpret_cast<const float2*>(sv + 16 * RV + 4 * (8 * nt + 2 * tig));
        float v0 = gk.x * (s[nt][0] + s[nt][2]) * inv_qs;
        float v1 = gk.y * (s[nt][1] + s[nt][3]) * inv_qs;
        if constexpr (QJL) {
          const float2 rh = *reinterpret_cast<const float2*>(sk + 16 * RK + 64 + 256 + 4 * (8 * nt + 2 * tig));
          v0 += a.qjl_coef * rh.x * (sq[nt][0] + sq[nt][2]) * inv_us;
          v1 += a.qjl_coef * rh.y * (sq[nt][1] + sq[nt][3]) * inv_us;
        }
        const int tt = t0 + 8 * nt + 2 * tig;
        u[2 * nt] = tt < ctx ? v0 : -INFINITY;
        u[2 * nt + 1] = tt + 1 < ctx ? v1 : -INFINITY;
        wv[2 * nt] = gv.x;
        wv[2 * nt + 1] = gv.y;
      }
      uint32_t bp0, bp1;
      float W0, W1;
      softmax_block(st, u, wv, lane, tig, bp0, bp1, W0, W1, false);

      // acc^T += V_hat^T P'^T, per m-tile of 16 coordinates
      uint32_t vA[2], vB[2], vC[2], vD[2];
      load_sixteenth<BV>(sv + (2 * tig) * RV, g_, vA);
      load_sixteenth<BV>(sv + (2 * tig + 1) * RV, g_, vB);
      load_sixteenth<BV>(sv + (2 * tig + 8) * RV, g_, vC);
      load_sixteenth<BV>(sv + (2 * tig + 9) * RV, g_, vD);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t xab[2] = {prmt(vA[half], vB[half], 0x5140u), prmt(vA[half], vB[half], 0x7362u)};
        const uint32_t xcd[2] = {prmt(vC[half], vD[half], 0x5140u), prmt(vC[half], vD[half], 0x7362u)};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int mt = 4 * half + m;
          const uint32_t nab = (m & 1) ? (xab[m >> 1] >> 16) : (xab[m >> 1] & 0xFFFFu);
          const uint32_t ncd = (m & 1) ? (xcd[m >> 1] >> 16) : (xcd[m >> 1] & 0xFFFFu);
          uint32_t lo, hi, lo2, hi2;
          lookup4<BV>(nab, tv, lo, hi);
          lookup4<BV>(ncd, tv, lo2, hi2);
          const uint32_t av[4] = {prmt(lo, hi, 0x6240u), prmt(lo, hi, 0x7351u), prmt(lo2, hi2, 0x6240u),
                                  prmt(lo2, hi2, 0x7351u)};
          float dv[4];
          mma_f16(dv, av, bp0, bp1, zero4);
          st.acc[mt][0] = fmaf(W0, dv[0], st.acc[mt][0]);
          st.acc[mt][1] = fmaf(W1, dv[1], st.acc[mt][1]);
          st.acc[mt][2] = fmaf(W0, dv[2], st.acc[mt][2]);
          st.acc[mt][3] = fmaf(W1, dv[3], st.acc[mt][3]);
        }
      }
    }
    __syncwarp();
    if (i + kStages < n_my) {
      if (issue_block(ring, stage, a, b, kvh, j + kWarps * kStages, lane)) valid_mask |= 1u << stage;
      else valid_mask &= ~(1u << stage);
    }
  }
  if (aborted) {  // drain copies still in flight into this warp's ring before leaving it
    for (int k = i + 1; k < n_my && k < i + kStages; ++k) mbar_wait(ring.bar + (k % kStages), (uint32_t)(k / kStages) & 1u);
    st.M = -INFINITY;
  }
  __syncthreads();
  write_partials(st, reinterpret_cast<float*>(smem_raw), warp, lane, gc, a, b, head0, split);
}

// ------------------------------------------------------- bf16 decode kernel

__global__ void __launch_bounds__(kWarps * 32) k_decode_bf16(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int RB = kD * 2;  // bytes per token row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_ = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.ngroups, hg = blockIdx.y % a.ngroups;
  const int b = blockIdx.z;
  const int head0 = kvh * a.g + hg * 8;
  const int gc = min(8, a.g - hg * 8);
  int ctx = __ldg(a.ctx_lens + b);
  if (ctx < 0 || ctx > a.max_blocks * kBlock) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_status(a.status, TQ_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : a.max_blocks * kBlock;
  }
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int j0 = (int)((int64_t)split * nblk / a.splits);
  const int j1 = (int)((int64_t)(split + 1) * nblk / a.splits);
  const int n_my = j1 - j0 > warp ? (j1 - j0 - warp + kWarps - 1) / kWarps : 0;
  constexpr int kSt = 3;
  const int stage_bytes = a.kpage + a.vpage;
  Ring ring;
  ring.stage_bytes = stage_bytes;
  ring.buf = smem_raw + warp * kSt * stage_bytes;
  ring.bar = reinterpret_cast<uint64_t*>(smem_raw + kWarps * kSt * stage_bytes) + warp * kSt;
  if (lane == 0)
    for (int s = 0; s < kSt; ++s) mbar_init(ring.bar + s, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  uint32_t valid_mask = 0u;
  for (int s = 0; s < kSt && s < n_my; ++s)
    if (issue_block(ring, s, a, b, kvh, j0 + warp + kWarps * s, lane)) valid_mask |= 1u << s;

  // bf16 query fragments: rows g_ = hi part, g_ + 8 = lo part of head g_
  const bool hv = g_ < gc;
  uint32_t aq[8][4];
  {
    float v[32];
    if (hv) load32<float>(a.qrot + ((int64_t)b * a.Hq + head0 + g_) * kD + 32 * tig, v);
    else
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        hi[k] = __bfloat162float(__float2bfloat16_rn(v[4 * c + k]));
        lo[k] = v[4 * c + k] - hi[k];
      }
      aq[c][0] = pack_bf162(hi[0], hi[1]);
      aq[c][1] = pack_bf162(lo[0], lo[1]);
      aq[c][2] = pack_bf162(hi[2], hi[3]);
      aq[c][3] = pack_bf162(lo[2], lo[3]);
    }
  }
  SoftmaxState st;
  st.M = -INFINITY;
  st.l = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.acc[i][0] = st.acc[i][1] = st.acc[i][2] = st.acc[i][3] = 0.0f;
  const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float ones[4] = {1.0f, 1.0f, 1.0f, 1.0f};
  int i = 0;
  bool aborted = false;
  for (; i < n_my; ++i) {
    const int stage = i % kSt;
    if (!mbar_wait(ring.bar + stage, (uint32_t)(i / kSt) & 1u)) {
      if (lane == 0) flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    const int j = j0 + warp + kWarps * i;
    if (valid_mask & (1u << stage)) {
      const uint8_t* sk = ring.buf + stage * stage_bytes;
      const uint8_t* sv = sk + a.kpage;
      const int t0 = j * kBlock;
      float u[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        // keys of token 8 nt + g_, coordinates [32 tig, 32 tig + 32): 64 contiguous bytes
        const uint4* kr = reinterpret_cast<const uint4*>(sk + (8 * nt + g_) * RB + 64 * tig);
        uint32_t kw[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint4 v = kr[x];
          kw[4 * x] = v.x; kw[4 * x + 1] = v.y; kw[4 * x + 2] = v.z; kw[4 * x + 3] = v.w;
        }
        float accs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < 8; ++c) mma_bf16(accs, aq[c], kw[2 * c], kw[2 * c + 1], accs);
        const int tt = t0 + 8 * nt + 2 * tig;
        u[2 * nt] = tt < ctx ? accs[0] + accs[2] : -INFINITY;
        u[2 * nt + 1] = tt + 1 < ctx ? accs[1] + accs[3] : -INFINITY;
      }
      uint32_t bp0, bp1, bl0, bl1;
      float W0, W1;
      softmax_block(st, u, ones, lane, tig, bp0, bp1, W0, W1, true, &bl0, &bl1);
      // values: rows = coordinates 16 g_ + 2i (+1), k = tokens 2tig, 2tig+1, 2tig+8, 2tig+9
      const uint4* va = reinterpret_cast<const uint4*>(sv + (2 * tig) * RB + 32 * g_);
      const uint4* vb = reinterpret_cast<const uint4*>(sv + (2 * tig + 1) * RB + 32 * g_);
      const uint4* vc = reinterpret_cast<const uint4*>(sv + (2 * tig + 8) * RB + 32 * g_);
      const uint4* vd = reinterpret_cast<const uint4*>(sv + (2 * tig + 9) * RB + 32 * g_);
      uint32_t wa[8], wb[8], wc[8], wd[8];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        uint4 t;
        t = va[x]; wa[4 * x] = t.x; wa[4 * x + 1] = t.y; wa[4 * x + 2] = t.z; wa[4 * x + 3] = t.w;
        t = vb[x]; wb[4 * x] = t.x; wb[4 * x + 1] = t.y; wb[4 * x + 2] = t.z; wb[4 * x + 3] = t.w;
        t = vc[x]; wc[4 * x] = t.x; wc[4 * x + 1] = t.y; wc[4 * x + 2] = t.z; wc[4 * x + 3] = t.w;
        t = vd[x]; wd[4 * x] = t.x; wd[4 * x + 1] = t.y; wd[4 * x + 2] = t.z; wd[4 * x + 3] = t.w;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t av[4] = {prmt(wa[mt], wb[mt], 0x5410u), prmt(wa[mt], wb[mt], 0x7632u),
                                prmt(wc[mt], wd[mt], 0x5410u), prmt(wc[mt], wd[mt], 0x7632u)};
        float dv[4], dl[4];
        mma_bf16(dv, av, bp0, bp1, zero4);
        mma_bf16(dl, av, bl0, bl1, zero4);
        st.acc[mt][0] = fmaf(W0, dv[0] + dl[0], st.acc[mt][0]);
        st.acc[mt][1] = fmaf(W1, dv[1] + dl[1], st.acc[mt][1]);
        st.acc[mt][2] = fmaf(W0, dv[2] + dl[2], st.acc[mt][2]);
        st.acc[mt][3] = fmaf(W1, dv[3] + dl[3], st.acc[mt][3]);
      }
    }
    __syncwarp();
    if (i + kSt < n_my) {
      if (issue_block(ring, stage, a, b, kvh, j + kWarps * kSt, lane)) valid_mask |= 1u << stage;
      else valid_mask &= ~(1u << stage);
    }
  }
  if (aborted) {
    for (int k = i + 1; k < n_my && k < i + kSt; ++k) mbar_wait(ring.bar + (k % kSt), (uint32_t)(k / kSt) & 1u);
    st.M = -INFINITY;
  }
  __syncthreads();
  write_partials(st, reinterpret_cast<float*>(smem_raw), warp, lane, gc, a, b, head0, split);
}

// ------------------------------------------------------------- prologue

enum { ROTQ_IDENTITY = 0, ROTQ_HADAMARD = 1, ROTQ_DENSE = 2 };

// One warp per (sequence, query head).  qrot = Pi q * scale; uq = S qrot (QJL).
template <typename TQ>
__global__ void __launch_bounds__(128) k_rotate_q(const TQ* __restrict__ q, int64_t n_rows, int kind,
                                                  const float* __restrict__ rot, const float* __restrict__ S,
                                                  float scale, float* qrot, float* uq) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const TQ* src = q + row * kD;
  float x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = load_elem<TQ>(src + 4 * lane + k);
  float y[4];
  if (kind == ROTQ_HADAMARD) {
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = x[k] * __ldg(rot + 4 * lane + k);
    // bits 0, 1 of the coordinate inside the lane, bits 2..6 across lanes
    float a0 = y[0] + y[1], a1 = y[0] - y[1], a2 = y[2] + y[3], a3 = y[2] - y[3];
    y[0] = a0 + a2; y[2] = a0 - a2; y[1] = a1 + a3; y[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float o = __shfl_xor_sync(0xffffffffu, y[k], m);
        y[k] = upper ? (o - y[k]) : (y[k] + o);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] *= 0.08838834764831845f * scale;
  } else if (kind == ROTQ_DENSE) {
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = 0.0f;
    for (int j = 0; j < kD; ++j) {
      const float xj = __shfl_sync(0xffffffffu, x[j & 3], j >> 2);
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = fmaf(__ldg(rot + (4 * lane + k) * kD + j), xj, y[k]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] *= scale;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = x[k] * scale;
  }
  *reinterpret_cast<float4*>(qrot + row * kD + 4 * lane) = make_float4(y[0], y[1], y[2], y[3]);
  if (S) {
    float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int j = 0; j < kD; ++j) {
      const float yj = __shfl_sync(0xffffffffu, y[j & 3], j >> 2);
#pragma unroll
      for (int k = 0; k < 4; ++k) z[k] = fmaf(__ldg(S + (4 * lane + k) * kD + j), yj, z[k]);
    }
    *reinterpret_cast<float4*>(uq + row * kD + 4 * lane) = make_float4(z[0], z[1], z[2], z[3]);
  }
}

// ------------------------------------------------------------- combine

template <typename TO>
__global__ void __launch_bounds__(128) k_combine(const float* __restrict__ part, const float* __restrict__ ml,
                                                 int splits, int kind, const float* __restrict__ rot, TO* out) {
  __shared__ float sm[256], sl[256], y[kD];
  __shared__ float stot[2];
  const int t = threadIdx.x;
  const int64_t bh = blockIdx.x;
  float mx = -INFINITY;
  for (int s = t; s < splits; s += blockDim.x) mx = fmaxf(mx, ml[(bh * splits + s) * 2]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) sm[t >> 5] = mx;
  __syncthreads();
  if (t == 0) stot[0] = fmaxf(fmaxf(sm[0], sm[1]), fmaxf(sm[2], sm[3]));
  __syncthreads();
  const float M = stot[0];
  for (int s = t; s < splits; s += blockDim.x) {
    const float ms = ml[(bh * splits + s) * 2];
    const float f = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
    sm[s] = f;
    sl[s] = ml[(bh * splits + s) * 2 + 1] * f;
  }
  __syncthreads();
  float acc = 0.0f, L = 0.0f;
  for (int s = 0; s < splits; ++s) {
    acc = fmaf(part[(bh * splits + s) * kD + t], sm[s], acc);
    L += sl[s];
  }
  float v = L > 0.0f ? acc / L : 0.0f;
  if (kind == ROTQ_HADAMARD) {
    y[t] = v;
    __syncthreads();
    for (int h = 1; h < kD; h <<= 1) {
      float a = 0.0f, c = 0.0f;
      const bool lower = (t & h) == 0;
      if (lower) { a = y[t]; c = y[t + h]; }
      __syncthreads();
      if (lower) { y[t] = a + c; y[t + h] = a - c; }
      __syncthreads();
    }
    v = y[t] * 0.08838834764831845f * __ldg(rot + t);
  } else if (kind == ROTQ_DENSE) {
    y[t] = v;
    __syncthreads();
    float o = 0.0f;
    for (int i = 0; i < kD; ++i) o = fmaf(__ldg(rot + i * kD + t), y[i], o);  // (Pi^T y)_t
    v = o;
  }
  store_elem<TO>(out + bh * kD + t, v);
}

// ------------------------------------------------------------- launcher

Codebook codebook_of(const tq_cache_desc& d, int which);

template <int BK, int BV, bool QJL>
static cudaError_t run_packed(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = k_decode_packed<BK, BV, QJL>;
  size_t smem = (size_t)kWarps * kStages * (a.kpage + a.vpage) + kWarps * kStages * 8;
  const size_t red = (size_t)(kWarps * 8 * kD + 2 * kWarps * 8) * 4;
  if (smem < red) smem = red;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

template <int BK, bool QJL>
static cudaError_t dispatch_bv(const DecodeArgs& a, int bv, dim3 grid, cudaStream_t st) {
  switch (bv) {
    case 2: return run_packed<BK, 2, QJL>(a, grid, st);
    case 3: return run_packed<BK, 3, QJL>(a, grid, st);
    default: return run_packed<BK, 4, QJL>(a, grid, st);
  }
}

cudaError_t launch_decode(const DecodeCall& c, cudaStream_t st) {
  const tq_cache_desc& d = *c.desc;
  const bool bf16 = d.fmt.kv_format == TQ_KV_BF16;
  const bool qjl = !bf16 && d.fmt.qjl_k;
  const DecodeWorkspace ws = decode_workspace(c.batch, c.num_q_heads, c.splits, kD, qjl);
  float* qrot = reinterpret_cast<float*>(c.workspace + ws.qrot_off);
  float* uq = qjl ? qrot + (size_t)c.batch * c.num_q_heads * kD : nullptr;
  const int kind = bf16 ? ROTQ_IDENTITY : (d.fmt.rot_kind == TQ_ROT_DENSE ? ROTQ_DENSE : ROTQ_HADAMARD);
  const int64_t rows = (int64_t)c.batch * c.num_q_heads;
  const float scale = c.sm_scale * kLog2e;
  const unsigned rgrid = (unsigned)((rows + 3) / 4);
  if (c.q_dtype == TQ_F32)
    k_rotate_q<float><<<rgrid, 128, 0, st>>>(reinterpret_cast<const float*>(c.q), rows, kind, d.rotation,
                                             qjl ? d.qjl_proj : nullptr, scale, qrot, uq);
  else
    k_rotate_q<__nv_bfloat16><<<rgrid, 128, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(c.q), rows, kind,
                                                     d.rotation, qjl ? d.qjl_proj : nullptr, scale, qrot, uq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  DecodeArgs a;
  a.kpool = reinterpret_cast<const uint8_t*>(d.k_cache);
  a.vpool = reinterpret_cast<const uint8_t*>(d.v_cache);
  a.kpage = (int)page_bytes_of(d, 0);
  a.vpage = (int)page_bytes_of(d, 1);
  a.Hkv = d.num_kv_heads;
  a.num_blocks = d.num_blocks;
  a.block_table = c.block_table;
  a.max_blocks = c.max_blocks;
  a.ctx_lens = c.ctx_lens;
  a.qrot = qrot;
  a.uqjl = uq;
  a.Hq = c.num_q_heads;
  a.g = c.num_q_heads / d.num_kv_heads;
  a.ngroups = (a.g + 7) / 8;
  a.splits = c.splits;
  a.part = reinterpret_cast<float*>(c.workspace + ws.part_off);
  a.ml = reinterpret_cast<float*>(c.workspace + ws.ml_off);
  a.cbk = codebook_of(d, 0);
  a.cbv = codebook_of(d, 1);
  a.qjl_coef = 1.2533141373155003f / (float)kD;  // sqrt(pi/2) / m
  a.status = c.status;
  dim3 grid((unsigned)c.splits, (unsigned)(d.num_kv_heads * a.ngroups), (unsigned)c.batch);
  if (bf16) {
    size_t smem = (size_t)kWarps * 3 * (a.kpage + a.vpage) + kWarps * 3 * 8;
    e = cudaFuncSetAttribute(k_decode_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_decode_bf16<<<grid, kWarps * 32, smem, st>>>(a);
  } else {
    const int bk = d.fmt.bits_k, bv = d.fmt.bits_v;
    if (qjl) {
      switch (bk) {
        case 2: e = dispatch_bv<2, true>(a, bv, grid, st); break;
        case 3: e = dispatch_bv<3, true>(a, bv, grid, st); break;
        default: e = dispatch_bv<4, true>(a, bv, grid, st); break;
      }
    } else {
      switch (bk) {
        case 2: e = dispatch_bv<2, false>(a, bv, grid, st); break;
        case 3: e = dispatch_bv<3, false>(a, bv, grid, st); break;
        default: e = dispatch_bv<4, false>(a, bv, grid, st); break;
      }
    }
    if (e != cudaSuccess) return e;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned cgrid = (unsigned)rows;
  if (c.out_dtype == TQ_F32)
    k_combine<float><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, kind, d.rotation, reinterpret_cast<float*>(c.out));
  else
    k_combine<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, kind, d.rotation,
                                                    reinterpret_cast<__nv_bfloat16*>(c.out));
  return cudaGetLastError();
}

}  // namespace tq
