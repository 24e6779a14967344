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
//   k_rotate_q   warp per (sequence, query head): FWHT or dense mat-vec.
//   k_decode     one CTA per SM (16 warps; 8 for QJL keys and bf16 pages).  The context of every (sequence, KV
//                head, head group) unit is cut into `splits` equal chunks and
//                each warp owns one chunk: one balanced wave.  A warp streams
//                its blocks' K and V pages into its own 4-deep shared-memory
//                ring with 1-D bulk copies (cp.async.bulk, completion on an
//                mbarrier).  Codes become fp16 mma.sync m16n8k16 fragments
//                through byte-indexed tables in shared memory (one f16x2
//                entry per pair of codes, replicated per lane so lookups never
//                conflict): logits^T = Q'(16 rows = 8 heads x {hi, lo} fp16
//                split) x K_hat^T, then acc^T += V_hat^T x P'^T with
//                P'_t = 2^(u_t - M) gamma'_t / W_block (<= 1) and W_block
//                folded back in fp32.  At the end the warps of a CTA that share
//                a unit merge through shared memory and one partial is written.
//                bf16 layers use the same skeleton with bf16 MMAs on raw pages.
//   k_combine    CTA per (sequence, query head): log-sum-exp merge of the
//                chunks and the inverse rotation.
#include <cfloat>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kMaxStages = 4;
constexpr int kMaxFusedSplits = 128;  // the decode kernel merges its own chunks up to this split count
constexpr float kRescaleThreshold = 20.0f;  // log2 units before the running max is refreshed
constexpr float kLog2e = 1.4426950408889634f;
// P' = w / R * kPScale lies in (0, 2^14]: fp16 keeps 11 significant bits for
// every weight down to 2^-28 of the running maximum.
constexpr float kPScale = 16384.0f;

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

__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~1 s (returns false).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try(addr, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try(addr, parity)) return true;
    if ((it & 63) == 63 && global_ns() - t0 > 1000000000ull) return false;
  }
  return false;
}

// 2^x by the hardware approximation (relative error ~2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// The code tables sit at shared address kLutAddr = 0x10000 as 256 rows of 256 B
// (row e = pair byte e): bytes [0, 128) hold the key table's f16x2 entry once per
// lane, bytes [128, 256) the value table's.  The shared address of (row e, lane)
// is 0x10000 | e << 8 | lane * 4 (+128), so one byte permute of the code word
// with `lbase` = 0x10000 | lane * 4 (+128) gives the address directly.
constexpr uint32_t kLutAddr = 0x10000u;
constexpr uint32_t kLutBytes = 0x10000u;

__device__ __forceinline__ uint32_t lut(uint32_t lbase, uint32_t w, int k) {
  return lds32(__byte_perm(w, lbase, 0x7604u | ((uint32_t)k << 4)));
}

__device__ __forceinline__ uint32_t byte_of(uint32_t w, int k) { return __byte_perm(w, 0u, 0x4440u | (uint32_t)k); }

// ------------------------------------------------------- codes -> nibbles

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
// as 4 nibble words of 8 codes (byte k of word w = codes 8w + 2k, 8w + 2k + 1).
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
  int splits;  // chunks per unit
  int chunks;  // units * splits
  int stages;  // ring depth per warp
  int lut_shared;
  int smem_bytes;  // dynamic shared memory of the launch
  int fuse_combine;  // 0: k_combine finishes; 1: decode finishes (identity); 2: decode finishes (Hadamard)
  int* counters;     // [units] chunks finished per unit (zeroed by k_rotate_q)
  const float* rot;  // Hadamard signs (fuse_combine == 2)
  void* out;
  int out_bf16;
  float* part;  // [B][Hq][splits][d]
  float* ml;    // [B][Hq][splits][2]
  Codebook cbk, cbv;
  float qjl_coef;  // sqrt(pi/2) / m
  unsigned* status;
};

// Splits one fp32 query row (32 coordinates of quarter tig) into hi/lo A
// fragments of 8 k-chunks (fp16 with a power-of-two scale, or bf16).  Returns 1/scale.
template <bool BF16>
__device__ __forceinline__ float make_q_frags(const float* qrow, bool valid, int tig, uint32_t (&a)[8][4]) {
  float v[32];
  if (valid) {
    load32<float>(qrow + 32 * tig, v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  }
  float scale = 1.0f;
  if (!BF16) {
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
    mx = quad_max(mx);
    int e = 0;
    if (mx > 0.0f) frexpf(mx, &e);
    scale = ldexpf(1.0f, 14 - e);  // max |q| * scale < 2^14
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float s = v[4 * c + k] * scale;
      hi[k] = BF16 ? __bfloat162float(__float2bfloat16_rn(s)) : __half2float(__float2half_rn(s));
      lo[k] = s - hi[k];
    }
    if (BF16) {
      a[c][0] = pack_bf162(hi[0], hi[1]);
      a[c][1] = pack_bf162(lo[0], lo[1]);
      a[c][2] = pack_bf162(hi[2], hi[3]);
      a[c][3] = pack_bf162(lo[2], lo[3]);
    } else {
      a[c][0] = pack_half2(hi[0], hi[1]);
      a[c][1] = pack_half2(lo[0], lo[1]);
      a[c][2] = pack_half2(hi[2], hi[3]);
      a[c][3] = pack_half2(lo[2], lo[3]);
    }
  }
  return 1.0f / scale;
}

// Online-softmax state of one warp for head g_ (the thread's row): running max
// M of the base-2 logits, partial denominator l = sum 2^(u - M), and a running
// value reference R >= max_t 2^(u_t - M) gamma'_t.  The rotated-domain
// accumulator fragments acc[i] (columns = heads 2 tig, 2 tig + 1; rows = coords
// 16 g_ + 2i, +1) hold sum_t (2^(u_t - M) gamma'_t / R) c_V[idx'_t], so the MMA
// operand P' = 2^(u - M) gamma' / R never exceeds 1 in fp16 and the MMA
// accumulates straight into acc; the true sum is acc * R.
struct SoftmaxState {
  float M, l, R, rR;
  float acc[8][4];
};

// Given the 4 scaled logits u (tokens 2tig, 2tig+1, 8+2tig, 9+2tig) and value
// weights wv (gamma' or 1), updates M, l, R (rescaling acc when either moves)
// and returns the B fragments of P' (fp16, or bf16 hi + lo).
template <bool BF16>
__device__ __forceinline__ void softmax_block(SoftmaxState& st, const float (&u)[4], const float (&wv)[4], int tig,
                                              uint32_t& bp0, uint32_t& bp1, uint32_t& bl0, uint32_t& bl1) {
  // M is kept integral and R a power of two, so every rescale is exact and the
  // fp16 rounding of P' does not depend on which tokens came before.
  float bmax = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
  bmax = quad_max(bmax);
  if (__any_sync(0xffffffffu, bmax > st.M + kRescaleThreshold)) {
    const bool need = bmax > st.M + kRescaleThreshold;
    const float newM = need ? ceilf(bmax) : st.M;
    const float alpha = (st.M == -INFINITY) ? 0.0f : ldexpf(1.0f, (int)(st.M - newM));
    st.l *= alpha;
    st.R *= alpha;  // acc / R is unchanged by a common factor
    st.M = newM;
  }
  float w[4];
  float wmax = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float p = fast_exp2(u[e] - st.M);
    st.l += p;
    w[e] = p * wv[e];
    wmax = fmaxf(wmax, w[e]);
  }
  wmax = quad_max(wmax);
  if (__any_sync(0xffffffffu, wmax > st.R)) {
    // smallest power of two >= max(R, wmax)
    const float m = fmaxf(st.R, wmax);
    const float newR = m > 0.0f ? __uint_as_float((__float_as_uint(m) + 0x007FFFFFu) & 0xFF800000u) : 0.0f;
    const float beta = newR > 0.0f ? st.R / newR : 1.0f;
    st.R = newR;
    st.rR = newR > 0.0f ? kPScale / newR : 0.0f;
    const float b0 = __shfl_sync(0xffffffffu, beta, (2 * tig) * 4);
    const float b1 = __shfl_sync(0xffffffffu, beta, (2 * tig + 1) * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.acc[i][0] *= b0; st.acc[i][1] *= b1; st.acc[i][2] *= b0; st.acc[i][3] *= b1;
    }
  }
  float pn[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) pn[e] = w[e] * st.rR;
  if (BF16) {
    bp0 = pack_bf162(pn[0], pn[1]);
    bp1 = pack_bf162(pn[2], pn[3]);
    const __nv_bfloat162 h0 = *reinterpret_cast<__nv_bfloat162*>(&bp0);
    const __nv_bfloat162 h1 = *reinterpret_cast<__nv_bfloat162*>(&bp1);
    bl0 = pack_bf162(pn[0] - __low2float(h0), pn[1] - __high2float(h0));
    bl1 = pack_bf162(pn[2] - __low2float(h1), pn[3] - __high2float(h1));
  } else {
    bp0 = pack_half2(pn[0], pn[1]);
    bp1 = pack_half2(pn[2], pn[3]);
    bl0 = bl1 = 0u;
  }
}

// Block-table entries of one warp's chunk, read 32 at a time into a register
// (lane k holds entry 32 r + k) with the next 32 already in flight, so issuing a
// copy never waits on a global load.  Indices must be requested in increasing order.
struct BlockIds {
  const int32_t* row;  // block table row + j0
  int n, round;
  int cur, nxt;
  __device__ __forceinline__ void init(const int32_t* p, int count, int lane) {
    row = p;
    n = count;
    round = 0;
    cur = lane < n ? __ldg(row + lane) : 0;
    nxt = 32 + lane < n ? __ldg(row + 32 + lane) : 0;
  }
  __device__ __forceinline__ int get(int k, int lane) {
    if ((k >> 5) != round) {  // warp-uniform
      ++round;
      cur = nxt;
      const int j = 32 * (round + 1) + lane;
      nxt = j < n ? __ldg(row + j) : 0;
    }
    return __shfl_sync(0xffffffffu, cur, k & 31);
  }
};

// Per-warp ring of (K page, V page) stages fed by bulk copies.
struct Ring {
  uint8_t* buf;   // stages x (kpage + vpage)
  uint64_t* bar;  // stages
  int stage_bytes;
};

// Issues the copies of block j of sequence b into `stage` (lane 0 only).
// Returns true (on every lane) if the block id was valid and copies were issued.
__device__ __forceinline__ bool issue_block(const Ring& r, int stage, const DecodeArgs& a, int blk, int kvh,
                                            int lane) {
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

// ------------------------------------------------------------ block compute

// One 16-token block of packed K/V for one warp.
template <int BK, int BV, bool QJL>
__device__ __forceinline__ void packed_block(SoftmaxState& st, const uint8_t* sk, const uint8_t* sv, int t0, int ctx,
                                             const uint32_t (&aq)[8][4], const uint32_t (&au)[8][4], float inv_qs,
                                             float inv_us, uint32_t lk, uint32_t lv, float qjl_coef, int g_,
                                             int tig) {
  constexpr int RK = 16 * BK, RV = 16 * BV;
  float s[2][4], sq[2][4];
  uint32_t kn[2][4];
  load_quarter<BK>(sk + g_ * RK, tig, kn[0]);
  load_quarter<BK>(sk + (8 + g_) * RK, tig, kn[1]);
  {
    // two independent accumulation chains per n-tile (even / odd k-chunks)
    float acc2[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc2[nt][p][e] = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t w = kn[nt][c >> 1];
        const int k0 = 2 * (c & 1);
        mma_f16(acc2[nt][c & 1], aq[c], lut(lk, w, k0), lut(lk, w, k0 + 1), acc2[nt][c & 1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = acc2[nt][0][e] + acc2[nt][1][e];
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
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
  float u[4], wv[4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float2 gk = *reinterpret_cast<const float2*>(sk + 16 * RK + 4 * (8 * nt + 2 * tig));
    const float2 gv = *reinterpret_cast<const float2*>(sv + 16 * RV + 4 * (8 * nt + 2 * tig));
    float v0 = gk.x * (s[nt][0] + s[nt][2]) * inv_qs;
    float v1 = gk.y * (s[nt][1] + s[nt][3]) * inv_qs;
    if constexpr (QJL) {
      const float2 rh = *reinterpret_cast<const float2*>(sk + 16 * RK + 64 + 256 + 4 * (8 * nt + 2 * tig));
      v0 += qjl_coef * rh.x * (sq[nt][0] + sq[nt][2]) * inv_us;
      v1 += qjl_coef * rh.y * (sq[nt][1] + sq[nt][3]) * inv_us;
    }
    const int tt = t0 + 8 * nt + 2 * tig;
    u[2 * nt] = tt < ctx ? v0 : -INFINITY;
    u[2 * nt + 1] = tt + 1 < ctx ? v1 : -INFINITY;
    wv[2 * nt] = gv.x;
    wv[2 * nt + 1] = gv.y;
  }
  uint32_t bp0, bp1, bl0, bl1;
  softmax_block<false>(st, u, wv, tig, bp0, bp1, bl0, bl1);

  // values: rows = coordinates 16 g_ + 2i (+1), k = tokens 2tig, 2tig+1, 2tig+8, 2tig+9
  uint32_t vA[2], vB[2], vC[2], vD[2];
  load_sixteenth<BV>(sv + (2 * tig) * RV, g_, vA);
  load_sixteenth<BV>(sv + (2 * tig + 1) * RV, g_, vB);
  load_sixteenth<BV>(sv + (2 * tig + 8) * RV, g_, vC);
  load_sixteenth<BV>(sv + (2 * tig + 9) * RV, g_, vD);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      // byte m of a nibble word holds codes (2m, 2m+1): m-tiles 4 half + 2 q2 + {0, 1}
      const uint32_t sel = q2 ? 0x7362u : 0x5140u;
      const uint32_t xab = __byte_perm(vA[half], vB[half], sel);  // A(m), B(m), A(m+1), B(m+1)
      const uint32_t xcd = __byte_perm(vC[half], vD[half], sel);
      // pair bytes (token-A code | token-B code << 4): low nibbles -> row g_, high nibbles -> row g_+8
      const uint32_t lab = (xab & 0x0F0F0F0Fu) | ((xab >> 4) & 0xF0F0F0F0u);
      const uint32_t hab = ((xab >> 4) & 0x0F0F0F0Fu) | ((xab >> 8) & 0xF0F0F0F0u);
      const uint32_t lcd = (xcd & 0x0F0F0F0Fu) | ((xcd >> 4) & 0xF0F0F0F0u);
      const uint32_t hcd = ((xcd >> 4) & 0x0F0F0F0Fu) | ((xcd >> 8) & 0xF0F0F0F0u);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int mt = 4 * half + 2 * q2 + m;
        const uint32_t av[4] = {lut(lv, lab, 2 * m), lut(lv, hab, 2 * m), lut(lv, lcd, 2 * m),
                                lut(lv, hcd, 2 * m)};
        mma_f16(st.acc[mt], av, bp0, bp1, st.acc[mt]);
      }
    }
  }
}

// One 16-token block of raw bf16 K/V for one warp.
__device__ __forceinline__ void bf16_block(SoftmaxState& st, const uint8_t* sk, const uint8_t* sv, int t0, int ctx,
                                           const uint32_t (&aq)[8][4], int g_, int tig) {
  constexpr int RB = kD * 2;  // bytes per token row
  const float ones[4] = {1.0f, 1.0f, 1.0f, 1.0f};
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
  softmax_block<true>(st, u, ones, tig, bp0, bp1, bl0, bl1);
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
    const uint32_t av[4] = {__byte_perm(wa[mt], wb[mt], 0x5410u), __byte_perm(wa[mt], wb[mt], 0x7632u),
                            __byte_perm(wc[mt], wd[mt], 0x5410u), __byte_perm(wc[mt], wd[mt], 0x7632u)};
    mma_bf16(st.acc[mt], av, bp0, bp1, st.acc[mt]);
    mma_bf16(st.acc[mt], av, bl0, bl1, st.acc[mt]);
  }
}

// ------------------------------------------------------------ decode kernel

// KIND 0: packed codes (BK, BV, QJL); KIND 1: bf16 pages.  NW warps per CTA, one
// CTA per SM holding all of the SM's shared memory.
// Shared layout (absolute shared addresses; base = start of the dynamic window):
//   packed: rings of warps [0, n_lo) in [base, 0x10000), code tables in
//           [0x10000, 0x20000), rings of the other warps from 0x20000;
//   bf16:   rings from base.  mbarriers at the top.  The merge scratch of the
//   epilogue reuses the rings above the tables (drained by then).
template <int KIND, int BK, int BV, bool QJL, int NW>
__global__ void __launch_bounds__(NW * 32, 1) k_decode(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_ = lane >> 2, tig = lane & 3;
  const int stage_bytes = a.kpage + a.vpage;
  const uint32_t ring_bytes = (uint32_t)(a.stages * stage_bytes);
  const uint32_t base = smem_u32(smem_raw);
  const uint32_t bars_addr = (base + (uint32_t)a.smem_bytes - (uint32_t)(NW * kMaxStages * 8)) & ~15u;
  const uint32_t lo0 = (base + 127u) & ~127u;
  const uint32_t n_lo = (KIND == 0 && kLutAddr > lo0) ? (kLutAddr - lo0) / ring_bytes : 0u;
  const uint32_t hi0 = KIND == 0 ? kLutAddr + kLutBytes : lo0;
  const uint32_t n_hi = bars_addr > hi0 ? (bars_addr - hi0) / ring_bytes : 0u;
  const uint32_t red_bytes = (uint32_t)(NW * 8 * kD + 2 * NW * 8 + NW) * 4u;
  const bool layout_ok = (KIND == 1 || (base <= kLutAddr && kLutAddr + kLutBytes <= bars_addr)) &&
                         n_lo + n_hi >= (uint32_t)NW && hi0 + red_bytes <= bars_addr;
  auto gen = [&](uint32_t addr) { return smem_raw + (addr - base); };

  if (!layout_ok && threadIdx.x == 0 && blockIdx.x == 0) flag_status(a.status, TQ_DEV_LAYOUT);

  // this warp's chunk: unit = (sequence, kv head, head group), split s of its context
  const int ch = blockIdx.x * NW + warp;
  const bool has = layout_ok && ch < a.chunks;
  const int unit = has ? ch / a.splits : -1;
  const int s = has ? ch - unit * a.splits : 0;
  const int per_b = a.Hkv * a.ngroups;
  const int b = has ? unit / per_b : 0;
  const int r = has ? unit - b * per_b : 0;
  const int kvh = r / a.ngroups, hg = r - (r / a.ngroups) * a.ngroups;
  const int head0 = kvh * a.g + hg * 8;
  const int gc = min(8, a.g - hg * 8);
  int ctx = has ? __ldg(a.ctx_lens + b) : 0;
  if (ctx < 0 || ctx > a.max_blocks * kBlock) {
    if (lane == 0 && s == 0 && r == 0) flag_status(a.status, TQ_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : a.max_blocks * kBlock;
  }
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int j0 = (int)((int64_t)s * nblk / a.splits);
  const int j1 = (int)((int64_t)(s + 1) * nblk / a.splits);
  const int n_my = has ? j1 - j0 : 0;

  Ring ring;
  ring.stage_bytes = stage_bytes;
  const uint32_t rw = (uint32_t)warp;
  ring.buf = gen(rw < n_lo ? lo0 + rw * ring_bytes : hi0 + (rw - n_lo) * ring_bytes);
  ring.bar = reinterpret_cast<uint64_t*>(gen(bars_addr)) + warp * kMaxStages;
  if (lane == 0)
    for (int k = 0; k < a.stages; ++k) mbar_init(ring.bar + k, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();  // this warp's barriers are ready

  // first copies go out before the tables are built, to overlap their latency
  BlockIds ids;
  ids.init(a.block_table + (int64_t)b * a.max_blocks + j0, n_my, lane);
  uint32_t valid_mask = 0u;
  for (int k = 0; k < a.stages && k < n_my; ++k)
    if (issue_block(ring, k, a, ids.get(k, lane), kvh, lane)) valid_mask |= 1u << k;

  if constexpr (KIND == 0) {
    if (layout_ok) {
      // row e (pair byte, low nibble first) = f16x2(c[e & 15], c[e >> 4]), once per lane, K then V;
      // lanes 0..15 hold the key centroids, lanes 16..31 the value centroids
      constexpr uint32_t MK = (1u << BK) - 1u, MV = (1u << BV) - 1u;
      const float cl = lane < 16 ? a.cbk.c[lane & MK] : a.cbv.c[(lane - 16) & MV];
      uint32_t* tab = reinterpret_cast<uint32_t*>(gen(kLutAddr));
      for (int i = threadIdx.x; i < 256 * 64; i += blockDim.x) {
        const int e = i >> 6;              // warp-uniform
        const int vo = (i & 32) ? 16 : 0;  // warp-uniform
        const float lo = __shfl_sync(0xffffffffu, cl, vo + (e & 15));
        const float hi = __shfl_sync(0xffffffffu, cl, vo + (e >> 4));
        tab[i] = pack_half2(lo, hi);
      }
    }
  }
  __syncthreads();  // tables ready

  const bool hv = g_ < gc;
  const int64_t qrow = ((int64_t)b * a.Hq + head0 + (hv ? g_ : 0)) * kD;
  uint32_t aq[8][4];
  uint32_t au[8][4];
  float inv_qs = 1.0f, inv_us = 0.0f;
  inv_qs = make_q_frags<KIND == 1>(a.qrot + qrow, hv && has, tig, aq);
  if constexpr (QJL) inv_us = make_q_frags<false>(a.uqjl + qrow, hv && has, tig, au);
  const uint32_t lk = kLutAddr | (4u * lane);
  const uint32_t lv = lk + 128u;

  SoftmaxState st;
  st.M = -INFINITY;
  st.l = 0.0f;
  st.R = 0.0f;
  st.rR = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.acc[i][0] = st.acc[i][1] = st.acc[i][2] = st.acc[i][3] = 0.0f;

  int i = 0, stage = 0;
  uint32_t phase = 0u;
  bool aborted = false;
  for (; i < n_my; ++i) {
    if (!mbar_wait(ring.bar + stage, phase)) {
      if (lane == 0) flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    if (valid_mask & (1u << stage)) {
      const uint8_t* sk = ring.buf + stage * stage_bytes;
      const uint8_t* sv = sk + a.kpage;
      const int t0 = (j0 + i) * kBlock;
      if constexpr (KIND == 0)
        packed_block<BK, BV, QJL>(st, sk, sv, t0, ctx, aq, au, inv_qs, inv_us, lk, lv, a.qjl_coef, g_, tig);
      else
        bf16_block(st, sk, sv, t0, ctx, aq, g_, tig);
    }
    __syncwarp();
    if (i + a.stages < n_my) {
      if (issue_block(ring, stage, a, ids.get(i + a.stages, lane), kvh, lane)) valid_mask |= 1u << stage;
      else valid_mask &= ~(1u << stage);
    }
    if (++stage == a.stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if (aborted) {  // drain copies still in flight into this warp's ring before the smem is reused
    int stg = stage;
    uint32_t ph = phase;
    for (int k = i; k < n_my && k < i + a.stages; ++k) {
      mbar_wait(ring.bar + stg, ph);
      if (++stg == a.stages) { stg = 0; ph ^= 1u; }
    }
    st.M = -INFINITY;
    st.l = 0.0f;
  }

  // ---- merge the warps of this CTA that share a unit; one partial per group
  st.l = quad_sum(st.l);
  {  // acc holds sum / R per column (head): restore the scale
    const float r0 = __shfl_sync(0xffffffffu, st.R, (2 * tig) * 4) * (1.0f / kPScale);
    const float r1 = __shfl_sync(0xffffffffu, st.R, (2 * tig + 1) * 4) * (1.0f / kPScale);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= r0; st.acc[mt][1] *= r1; st.acc[mt][2] *= r0; st.acc[mt][3] *= r1;
    }
  }
  __syncthreads();  // every ring is drained: reuse the stage memory
  float* racc = reinterpret_cast<float*>(gen(hi0));  // [NW warps][8 heads][128]
  float* rm = racc + NW * 8 * kD;                     // [NW][8]
  float* rl = rm + NW * 8;                            // [NW][8]
  int* runit = reinterpret_cast<int*>(rl + NW * 8);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int c0 = 16 * g_ + 2 * mt;
    float* base = racc + warp * 8 * kD;
    base[(2 * tig) * kD + c0] = st.acc[mt][0];
    base[(2 * tig + 1) * kD + c0] = st.acc[mt][1];
    base[(2 * tig) * kD + c0 + 1] = st.acc[mt][2];
    base[(2 * tig + 1) * kD + c0 + 1] = st.acc[mt][3];
  }
  if (tig == 0) {
    rm[warp * 8 + g_] = st.M;
    rl[warp * 8 + g_] = st.l;
  }
  if (lane == 0) runit[warp] = unit;
  __syncthreads();
  if (!has) return;
  const bool leader = warp == 0 || runit[warp - 1] != unit;
  if (!leader) return;
  int wend = warp + 1;
  while (wend < NW && runit[wend] == unit) ++wend;
  const int covered = wend - warp;  // chunks s .. s + covered - 1 of this unit
  for (int h = 0; h < gc; ++h) {
    if (lane > 0 && lane < covered) {  // merged into slot s: mark the group's other slots empty
      const int64_t row2 = ((int64_t)b * a.Hq + head0 + h) * a.splits + s + lane;
      a.ml[row2 * 2] = -INFINITY;
      a.ml[row2 * 2 + 1] = 0.0f;
    }
    float Mt = -INFINITY;
    for (int w = warp; w < wend; ++w) Mt = fmaxf(Mt, rm[w * 8 + h]);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float L = 0.0f;
    for (int w = warp; w < wend; ++w) {
      const float mw = rm[w * 8 + h];
      const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - Mt);
      const float4 v = *reinterpret_cast<const float4*>(racc + (w * 8 + h) * kD + 4 * lane);
      acc[0] = fmaf(v.x, f, acc[0]);
      acc[1] = fmaf(v.y, f, acc[1]);
      acc[2] = fmaf(v.z, f, acc[2]);
      acc[3] = fmaf(v.w, f, acc[3]);
      L = fmaf(rl[w * 8 + h], f, L);
    }
    const int64_t row = ((int64_t)b * a.Hq + head0 + h) * a.splits + s;
    *reinterpret_cast<float4*>(a.part + row * kD + 4 * lane) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (lane == 0) {
      a.ml[row * 2] = Mt;
      a.ml[row * 2 + 1] = L;
    }
  }
  if (!a.fuse_combine) return;

  // ---- the warp that completes a unit merges its chunks and applies Pi^T
  __threadfence();
  int last = 0;
  if (lane == 0) last = atomicAdd(a.counters + unit, covered) + covered == a.splits;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // (max, denominator) of every (head, slot): lane l holds slots l + 32 g, all loads in flight at once
  constexpr int kG = kMaxFusedSplits / 32;
  const int64_t row0 = ((int64_t)b * a.Hq + head0) * a.splits;
  float fm[8][kG], fl[8][kG];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const int s2 = lane + 32 * g;
      const bool in = h < gc && s2 < a.splits;
      fm[h][g] = in ? __ldcg(a.ml + (row0 + (int64_t)h * a.splits + s2) * 2) : -INFINITY;
      fl[h][g] = in ? __ldcg(a.ml + (row0 + (int64_t)h * a.splits + s2) * 2 + 1) : 0.0f;
    }
  float Lh[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int g = 0; g < kG; ++g) mx = fmaxf(mx, fm[h][g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float L = 0.0f;
#pragma unroll
    for (int g = 0; g < kG; ++g) {  // fm becomes the slot weight
      fm[h][g] = fm[h][g] == -INFINITY ? 0.0f : exp2f(fm[h][g] - mx);
      L = fmaf(fl[h][g], fm[h][g], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    Lh[h] = L;
  }
  // sum the few non-empty slots (emptiness is per chunk, the same for every head)
  float yh[8][4];
#pragma unroll
  for (int h = 0; h < 8; ++h) yh[h][0] = yh[h][1] = yh[h][2] = yh[h][3] = 0.0f;
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    uint32_t live = __ballot_sync(0xffffffffu, fm[0][g] > 0.0f);
    while (live) {
      const int src = __ffs(live) - 1;
      live &= live - 1;
      const int s2 = src + 32 * g;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float f = __shfl_sync(0xffffffffu, fm[h][g], src);
        if (h < gc) {
          const float4 v =
              __ldcg(reinterpret_cast<const float4*>(a.part + (row0 + (int64_t)h * a.splits + s2) * kD) + lane);
          yh[h][0] = fmaf(v.x, f, yh[h][0]);
          yh[h][1] = fmaf(v.y, f, yh[h][1]);
          yh[h][2] = fmaf(v.z, f, yh[h][2]);
          yh[h][3] = fmaf(v.w, f, yh[h][3]);
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h >= gc) break;
    const float rl = Lh[h] > 0.0f ? 1.0f / Lh[h] : 0.0f;
    float y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = yh[h][k] * rl;
    if (a.fuse_combine == 2) {  // Hadamard: Pi^T y = D H y / sqrt(d); lane holds coordinates 4 lane + k
      float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
      y[0] = t0 + t2; y[2] = t0 - t2; y[1] = t1 + t3; y[3] = t1 - t3;
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
      for (int k = 0; k < 4; ++k) y[k] *= 0.08838834764831845f * __ldg(a.rot + 4 * lane + k);
    }
    const int64_t orow = ((int64_t)b * a.Hq + head0 + h) * kD + 4 * lane;
    if (a.out_bf16) {
      uint2 pk = make_uint2(pack_bf162(y[0], y[1]), pack_bf162(y[2], y[3]));
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow) = pk;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + orow) = make_float4(y[0], y[1], y[2], y[3]);
    }
  }
}

// ------------------------------------------------------------- prologue

enum { ROTQ_IDENTITY = 0, ROTQ_HADAMARD = 1, ROTQ_DENSE = 2 };

// One warp per (sequence, query head).  qrot = Pi q * scale; uq = S qrot (QJL).
// Also zeroes the decode's per-unit chunk counters.
template <typename TQ>
__global__ void __launch_bounds__(128) k_rotate_q(const TQ* __restrict__ q, int64_t n_rows, int kind,
                                                  const float* __restrict__ rot, const float* __restrict__ S,
                                                  float scale, float* qrot, float* uq, int* counters, int n_counters) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_counters; i += gridDim.x * blockDim.x) counters[i] = 0;
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
  __shared__ float stot[4];
  const int t = threadIdx.x;
  const int64_t bh = blockIdx.x;
  float mx = -INFINITY;
  for (int s = t; s < splits; s += blockDim.x) mx = fmaxf(mx, ml[(bh * splits + s) * 2]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) stot[t >> 5] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(stot[0], stot[1]), fmaxf(stot[2], stot[3]));
  for (int s = t; s < splits; s += blockDim.x) {
    const float ms = ml[(bh * splits + s) * 2];
    const float f = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
    sm[s] = f;
    sl[s] = f > 0.0f ? ml[(bh * splits + s) * 2 + 1] * f : 0.0f;
  }
  __syncthreads();
  float acc = 0.0f, L = 0.0f;
  for (int s = 0; s < splits; ++s) {
    if (sm[s] == 0.0f) continue;  // empty chunk or merged into another slot: its acc is not written
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

// Warps per decode CTA (one CTA per SM): packed codes without QJL run 16 warps
// at 128 registers; the QJL variant and bf16 pages run 8 warps with more registers.
constexpr int kPackedWarps = 16;
constexpr int kWideWarps = 8;

template <int KIND, int BK, int BV, bool QJL>
static cudaError_t run_decode(DecodeArgs a, cudaStream_t st) {
  constexpr int NW = (KIND == 0 && !QJL) ? kPackedWarps : kWideWarps;
  auto kern = k_decode<KIND, BK, BV, QJL, NW>;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  a.smem_bytes = optin;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((a.chunks + NW - 1) / NW);
  kern<<<grid, NW * 32, (size_t)optin, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BK, bool QJL>
static cudaError_t dispatch_bv(const DecodeArgs& a, int bv, cudaStream_t st) {
  switch (bv) {
    case 2: return run_decode<0, BK, 2, QJL>(a, st);
    case 3: return run_decode<0, BK, 3, QJL>(a, st);
    default: return run_decode<0, BK, 4, QJL>(a, st);
  }
}

static bool same_table(const Codebook& x, const Codebook& y, int bx, int by) {
  if (bx != by) return false;
  for (int i = 0; i < (1 << bx); ++i)
    if (x.c[i] != y.c[i]) return false;
  return true;
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
  int* counters = reinterpret_cast<int*>(c.workspace + ws.cnt_off);
  const int n_counters = (int)rows;  // >= batch * kv heads * head groups
  if (c.q_dtype == TQ_F32)
    k_rotate_q<float><<<rgrid, 128, 0, st>>>(reinterpret_cast<const float*>(c.q), rows, kind, d.rotation,
                                             qjl ? d.qjl_proj : nullptr, scale, qrot, uq, counters, n_counters);
  else
    k_rotate_q<__nv_bfloat16><<<rgrid, 128, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(c.q), rows, kind,
                                                     d.rotation, qjl ? d.qjl_proj : nullptr, scale, qrot, uq,
                                                     counters, n_counters);
  count_launch();
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
  a.chunks = c.batch * d.num_kv_heads * a.ngroups * c.splits;
  a.part = reinterpret_cast<float*>(c.workspace + ws.part_off);
  a.ml = reinterpret_cast<float*>(c.workspace + ws.ml_off);
  a.cbk = codebook_of(d, 0);
  a.cbv = codebook_of(d, 1);
  a.lut_shared = (!bf16 && same_table(a.cbk, a.cbv, d.fmt.bits_k, d.fmt.bits_v)) ? 1 : 0;
  a.qjl_coef = 1.2533141373155003f / (float)kD;  // sqrt(pi/2) / m
  a.status = c.status;
  // the decode kernel finishes the job itself unless the inverse rotation is a dense mat-vec
  a.fuse_combine = (kind == ROTQ_DENSE || c.splits > kMaxFusedSplits) ? 0 : (kind == ROTQ_HADAMARD ? 2 : 1);
  a.counters = counters;
  a.rot = d.rotation;
  a.out = c.out;
  a.out_bf16 = c.out_dtype == TQ_BF16 ? 1 : 0;
  // ring depth: 4 stages; 3 when two code tables would not leave room for 2 CTAs per SM;
  // 2 for bf16 pages (8 KB per block, one CTA per SM)
  a.stages = bf16 ? 3 : 4;
  if (bf16) {
    e = run_decode<1, 4, 4, false>(a, st);
  } else {
    const int bk = d.fmt.bits_k, bv = d.fmt.bits_v;
    if (qjl) {
      switch (bk) {
        case 2: e = dispatch_bv<2, true>(a, bv, st); break;
        case 3: e = dispatch_bv<3, true>(a, bv, st); break;
        default: e = dispatch_bv<4, true>(a, bv, st); break;
      }
    } else {
      switch (bk) {
        case 2: e = dispatch_bv<2, false>(a, bv, st); break;
        case 3: e = dispatch_bv<3, false>(a, bv, st); break;
        default: e = dispatch_bv<4, false>(a, bv, st); break;
      }
    }
  }
  if (e != cudaSuccess) return e;
  if (a.fuse_combine) return cudaSuccess;
  const unsigned cgrid = (unsigned)rows;
  if (c.out_dtype == TQ_F32)
    k_combine<float><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, kind, d.rotation, reinterpret_cast<float*>(c.out));
  else
    k_combine<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, kind, d.rotation,
                                                    reinterpret_cast<__nv_bfloat16*>(c.out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace tq
