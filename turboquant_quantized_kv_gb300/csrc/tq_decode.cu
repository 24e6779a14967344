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
//   k_rotate_q   warp per (sequence, query head): dense mat-vec or S q' (dense and
//                QJL layers only; Hadamard layers rotate the query inside k_decode).
//   k_decode     one CTA per SM (16 warps for groups of <= 4 query heads, also with
//                QJL keys; 12 for groups of 8 and FP8 keys; 8 for QJL keys with
//                groups of 8 and for bf16 pages).  The
//                block-table row of every (sequence, KV head, head group) unit is
//                cut into `splits` equal chunks (the context instead, when the row
//                is much wider than it) and each warp owns one chunk: one balanced
//                wave.  A warp streams its chunk's K and V pages into its
//                own ring of shared-memory stages (two 16-token blocks per stage)
//                with 16-byte cp.async copies, one stage ahead of the one it
//                computes on.  Codes become fp16 mma.sync m16n8k16 fragments
//                through byte-indexed tables in shared memory (one f16x2 entry per
//                pair of codes, replicated per lane so lookups never conflict):
//                logits = K_hat (16 tokens) x Q'^T (4 heads x {hi, lo} fp16 split),
//                online softmax in base 2, then acc += V_hat^T x P' in the rotated
//                domain.  At the end the warps of a CTA that share a unit merge
//                through shared memory and one partial per (unit, head) goes to the
//                workspace; the CTA that completes a unit (an acq_rel counter)
//                merges the unit's partials and applies Pi^T, one warp per head
//                row.  bf16 layers use the same skeleton with bf16 MMAs on raw pages.
//   k_combine    CTA per (sequence, query head): log-sum-exp merge of the chunks and
//                the inverse rotation, when the decode kernel cannot finish the job
//                itself (dense Pi, more than 128 splits).

#include <cuda_fp8.h>

#include <cfloat>

#include "tq_async.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kMaxFusedSplits = 128;  // the decode kernel merges its own chunks up to this split count
constexpr float kRescaleThreshold = 20.0f;  // log2 units before the running max is refreshed
constexpr float kLog2e = 1.4426950408889634f;
// P' = w / R * kPScale lies in (0, 2^14]: fp16 keeps 11 significant bits for
// every weight down to 2^-28 of the running maximum.
constexpr float kPScale = 16384.0f;

// ------------------------------------------------------------ PTX wrappers

// 2^k for an integer k, exactly (0 below the normal range, 2^127 above it).
__device__ __forceinline__ float pow2i(int k) {
  if (k < -126) return 0.0f;
  return __uint_as_float((uint32_t)(min(k, 127) + 127) << 23);
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

// Two FP8 E4M3 values (low byte first) as an f16x2 word (exact: E4M3 is a subset of fp16).
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

__device__ __forceinline__ uint32_t lut(uint32_t lbase, uint32_t w, int k) {
  return lds32(__byte_perm(w, lbase, 0x7604u | ((uint32_t)k << 4)));
}

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
  const float* qrot;  // [B][Hq][d] scaled rotated queries (q_in_kernel == 0)
  const float* uqjl;  // [B][Hq][d] S q' (QJL only)
  const void* q;      // [B][Hq][d] raw queries (q_in_kernel != 0; 16-byte aligned rows)
  int q_bf16;
  int q_in_kernel;    // 0: read qrot; 1: rotate q here (Hadamard); 2: scale q here (no rotation)
  float q_scale;      // sm_scale * log2 e
  int pdl;            // host side: launched as a programmatic dependent of the previous kernel
  int overlap_append;  // 1: follows this library's append (directly or through the query pass): wait before the first page copy
  int Hq, g, ngroups;
  int splits;  // chunks per unit
  int chunks;  // units * splits
  int smem_bytes;  // dynamic shared memory of the launch
  int fuse_combine;  // 0: k_combine finishes; the decode finishes with 1: identity, 2: Hadamard, 3: dense Pi^T
  int* counters;     // [units] chunks finished per unit (zeroed by k_rotate_q)
  const float* rot;  // Hadamard signs (fuse_combine == 2)
  void* out;
  int out_bf16;
  float* part;  // [B][Hq][splits][d]
  float* ml;    // [B][Hq][splits][2]
  Codebook cbk, cbv;
  float qjl_coef;  // sqrt(pi/2) / m
  unsigned* status;
  // tq_decode_step (packed Hadamard layers without QJL): the new token of sequence b,
  // [B][Hkv][d] each, written by the warp that holds block (ctx_b - 1) / 16 of its unit
  const void* new_k;
  const void* new_v;
  int new_bf16;
  int norm_raw;  // TQ_NORM_RAW: gamma = n
};

// One new vector quantized by a whole warp (tq_decode_step): lane l holds x_j for
// j = 4 l .. 4 l + 3.  y = H D x / (sqrt(d) n) with n = ||x||, code_j = #{k : y_j >=
// beta_k} (ties go up; y = 0 for the zero vector, so its codes are 2^(b-1) and gamma
// 0), gamma = n / ||c[code]|| (n with TQ_NORM_RAW).  On return lane w < 4 BITS holds
// word w of the LSB-first record (code j in bits BITS j .. BITS j + BITS - 1).
template <int BITS>
__device__ __forceinline__ void warp_quantize_record(const float (&x)[4], const float4& sg, const Codebook& cb,
                                                     bool norm_raw, int lane, uint32_t& word, float& gamma) {
  float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float n = sqrtf(ss);
  float y[4] = {x[0] * sg.x, x[1] * sg.y, x[2] * sg.z, x[3] * sg.w};
  {  // bits 0, 1 of the coordinate in the lane, bits 2..6 across lanes
    const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
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
  }
  const float inv = n > 0.0f ? 0.08838834764831845f / n : 0.0f;  // 1 / (sqrt(128) n)
  constexpr int NB = (1 << BITS) - 1;
  uint32_t f = 0u;
  float c2 = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float yk = y[k] * inv;
    uint32_t c = 0u;  // #{t : y >= beta_t} by bisection (the boundaries ascend)
#pragma unroll
    for (int step = 1 << (BITS - 1); step > 0; step >>= 1)
      if (yk >= cb.b[c + step - 1]) c += step;
    const float ck = cb.c[c];
    c2 = fmaf(ck, ck, c2);
    f |= c << (BITS * k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c2 += __shfl_xor_sync(0xffffffffu, c2, o);
  gamma = norm_raw ? n : ((n > 0.0f && c2 > 0.0f) ? n / sqrtf(c2) : 0.0f);
  // the lane's 4 BITS bits sit at bit 4 BITS l of the record: words w0 and maybe w0 + 1
  const int o = 4 * BITS * lane, w0 = o >> 5, sh = o & 31;
  const uint32_t lo = f << sh, hi = sh + 4 * BITS > 32 ? f >> (32 - sh) : 0u;
  word = 0u;
#pragma unroll
  for (int w = 0; w < 4 * BITS; ++w) {
    const uint32_t r = __reduce_or_sync(0xffffffffu, (w == w0 ? lo : 0u) | (w == w0 + 1 ? hi : 0u));
    if (lane == w) word = r;
  }
}

// Lane layout of a warp (g_ = lane / 4, tig = lane % 4) for NT n-tiles of 4 heads.
//
// Keys: logits = K_hat (16 tokens x 16 coordinates) x Q'^T (16 x 8) per k-chunk c:
// A rows are tokens g_, g_ + 8 of the block; the k index 2 tig + e maps to
// coordinate 32 tig + 4 c + e and 2 tig + 8 + e to 32 tig + 4 c + 2 + e, so a
// lane's A entries are the code bytes 16 tig + 2c, 2c + 1 of its two records.
// Column n = 2 h + part (part 0: fp16 hi of the query, 1: the lo remainder), so
// the lane holding D gets head 4 nt + tig for tokens g_ and g_ + 8.
//
// Values: acc (32 coordinates x 8 columns) += A (16 coordinate pairs x 16) x B
// per m-tile mt and token tile kt, with k = (position p, parity e) and a block-
// diagonal B[(p, e)][(h, e')] = P'[h][token(p)] [e = e'].  A[(row j)][(p, e)] is
// the code pair byte of token(p), so bytes are used as stored.  Row g_ of m-tile
// mt is the lane's byte 2 mt of coordinates [16 g_, 16 g_ + 16), row g_ + 8 byte
// 2 mt + 1; position p = tig of tile kt is token ta(tig) + 8 kt and p = tig + 4 is
// token tb(tig) + 8 kt, where {ta, tb} = {2 tig, 2 tig + 1} with ta odd for odd tig:
// the four records one load instruction reads then alternate between the two
// 64-byte halves of a 128-byte bank line (fewer shared-memory bank conflicts).
// The lane holding D gets head 4 nt + tig at coordinates 16 g_ + 4 mt + {0, 1, 2, 3}
// = acc[nt][mt][0..3].
__device__ __forceinline__ int tok_a(int tig) { return 2 * tig + (tig & 1); }
__device__ __forceinline__ int tok_b(int tig) { return 2 * tig + 1 - (tig & 1); }

// Key-side B fragments of one n-tile: lane (g_, tig) holds column g_ (head 4 nt +
// g_ / 2, part g_ & 1) at coordinates 32 tig + [0, 32) (v = the query row there):
// chunk c, b0 = {4c, 4c + 1}, b1 = {4c + 2, 4c + 3}.  fp16 with a power-of-two
// scale per head (max |q| scale < 2^14), or bf16.  Returns 1 / scale.
template <bool BF16>
__device__ __forceinline__ float make_q_frags(const float (&v)[32], int part, uint32_t (&bq)[8][2]) {
  float scale = 1.0f, inv_scale = 1.0f;
  if (!BF16) {
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
    mx = quad_max(mx);  // the quad (same g_) holds one head
    // mx in [2^(e-1), 2^e): scale = 2^(14 - e) (1 for a zero or subnormal row)
    const int ebits = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
    scale = ebits > 0 ? pow2i(140 - ebits) : 1.0f;
    inv_scale = ebits > 0 ? pow2i(ebits - 140) : 1.0f;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // pair (4c + 2j, 4c + 2j + 1): hi = round(s), lo = s - hi
      const float s0 = v[4 * c + 2 * j] * scale, s1 = v[4 * c + 2 * j + 1] * scale;
      uint32_t hi;
      float2 back;
      if (BF16) {
        hi = pack_bf162(s0, s1);
        back = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
      } else {
        hi = pack_half2(s0, s1);
        back = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      }
      const uint32_t lo = BF16 ? pack_bf162(s0 - back.x, s1 - back.y) : pack_half2(s0 - back.x, s1 - back.y);
      bq[c][j] = part ? lo : hi;
    }
  return inv_scale;
}

__device__ __forceinline__ void load_q(const float* qrow, bool valid, int tig, float (&v)[32]) {
  if (valid) {
    load32<float>(qrow + 32 * tig, v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  }
}

// Raw query coordinates 32 tig + [0, 32) of row `row` (fp32 or bf16).
__device__ __forceinline__ void load_q_raw(const void* q, bool bf16, int64_t row, bool valid, int tig,
                                           float (&v)[32]) {
  if (!valid) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  } else if (bf16) {
    load32<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(q) + row * kD + 32 * tig, v);
  } else {
    load32<float>(reinterpret_cast<const float*>(q) + row * kD + 32 * tig, v);
  }
}

// q' = scale * H (s * q) / sqrt(d) for a row spread over the 4 lanes of a quad (lane
// tig holds coordinates 32 tig + i): the Walsh-Hadamard butterflies of bits 0..4 run
// in registers, bits 5 and 6 across the quad.
__device__ __forceinline__ void rotate_q_quad(float (&v)[32], const float* signs, int tig, float scale) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= __ldg(signs + 32 * tig + i);
#pragma unroll
  for (int h = 1; h < 32; h <<= 1)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if ((i & h) == 0) {
        const float x = v[i], y = v[i + h];
        v[i] = x + y;
        v[i + h] = x - y;
      }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = (tig & m) ? (o - v[i]) : (v[i] + o);
    }
  const float f = scale * 0.08838834764831845f;
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= f;
}

// Online-softmax state of head 4 nt + tig, replicated on the 8 lanes of that tig:
// running max M (integral, base 2), this lane's share of l = sum 2^(u - M), and a
// power-of-two reference R >= every weight 2^(u - M) gamma' seen, so the fp16
// MMA operand P' = w kPScale / R stays in (0, kPScale].  acc holds
// sum_t P'_t c_V[idx'_t]; the true sum is acc R / kPScale.
template <int NT>
struct SoftmaxState {
  float M[NT], l[NT], R[NT], rR[NT];
  float acc[NT][4][4];
};

// Max over the 8 lanes sharing tig.
__device__ __forceinline__ float col_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}

__device__ __forceinline__ float col_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// u[nt][i]: base-2 logits of head 4 nt + tig for the lane's T tokens (pairs
// g_, g_ + 8 of T / 2 blocks; -inf when masked); wv[i]: their value weights
// (gamma' or 1; 0 when masked).  Updates the state and returns P' of each pair
// packed (fp16; bf16 hi in pk, lo in pl).
template <int NT, bool BF16, int T>
__device__ __forceinline__ void softmax_tokens(SoftmaxState<NT>& st, const float (&u)[NT][T], const float (&wv)[T],
                                               uint32_t (&pk)[NT][T / 2], uint32_t (&pl)[NT][T / 2]) {
  // M integral and R a power of two: every rescale is exact, and the rounding of
  // P' does not depend on the tokens that came before (split invariance).
  float um[NT];
  bool up = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    um[nt] = u[nt][0];
#pragma unroll
    for (int i = 1; i < T; ++i) um[nt] = fmaxf(um[nt], u[nt][i]);
    up |= um[nt] > st.M[nt] + kRescaleThreshold;
  }
  if (__any_sync(0xffffffffu, up)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float bm = col_max(um[nt]);
      if (bm > st.M[nt] + kRescaleThreshold) {  // the same on the head's lanes
        const float newM = ceilf(bm);
        const float alpha = (st.M[nt] == -INFINITY) ? 0.0f : pow2i((int)(st.M[nt] - newM));
        st.l[nt] *= alpha;
        st.R[nt] *= alpha;  // acc R is the true sum: scale R, keep acc
        st.rR[nt] = st.R[nt] > 0.0f ? kPScale / st.R[nt] : 0.0f;
        st.M[nt] = newM;
      }
    }
  }
  float w[NT][T];
  bool grow = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < T; ++i) {
      const float p = fast_exp2(u[nt][i] - st.M[nt]);
      st.l[nt] += p;
      w[nt][i] = p * wv[i];
      grow |= w[nt][i] > st.R[nt];
    }
  if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float wm = w[nt][0];
#pragma unroll
      for (int i = 1; i < T; ++i) wm = fmaxf(wm, w[nt][i]);
      wm = col_max(wm);
      if (wm > st.R[nt]) {
        const float newR = __uint_as_float((__float_as_uint(wm) + 0x007FFFFFu) & 0xFF800000u);  // pow2 >= wm
        const float beta = st.R[nt] / newR;
        st.R[nt] = newR;
        st.rR[nt] = kPScale / newR;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) st.acc[nt][mt][e] *= beta;
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < T / 2; ++j) {
      const float p0 = w[nt][2 * j] * st.rR[nt], p1 = w[nt][2 * j + 1] * st.rR[nt];
      if (BF16) {
        pk[nt][j] = pack_bf162(p0, p1);
        const __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&pk[nt][j]);
        pl[nt][j] = pack_bf162(p0 - __low2float(h), p1 - __high2float(h));
      } else {
        pk[nt][j] = pack_half2(p0, p1);
        pl[nt][j] = 0u;
      }
    }
}

// Value-side B fragments from the packed P' pairs: lane (g, t) takes head 4 nt + g/2
// at tokens ta(t), ta(t) + 8 (from lane 4 ta(t) + g/2) and tb(t), tb(t) + 8 (lane
// 4 tb(t) + g/2), each placed in half g & 1 of its pair (the other half 0).
struct PTranspose {
  int srcx, srcy;
  uint32_t sel0, sel1;  // byte selectors for token tile 0 (low halves) and 1 (high halves)
  __device__ __forceinline__ void init(int g_, int tig) {
    srcx = 4 * tok_a(tig) + (g_ >> 1);
    srcy = 4 * tok_b(tig) + (g_ >> 1);
    sel0 = (g_ & 1) ? 0x1044u : 0x4410u;
    sel1 = (g_ & 1) ? 0x3244u : 0x4432u;
  }
  __device__ __forceinline__ void apply(uint32_t pk, uint32_t (&bv)[2][2]) const {
    const uint32_t x = __shfl_sync(0xffffffffu, pk, srcx);
    const uint32_t y = __shfl_sync(0xffffffffu, pk, srcy);
    bv[0][0] = __byte_perm(x, 0u, sel0);
    bv[0][1] = __byte_perm(y, 0u, sel0);
    bv[1][0] = __byte_perm(x, 0u, sel1);
    bv[1][1] = __byte_perm(y, 0u, sel1);
  }
};

// Block-table entries of one warp's chunk, read 32 at a time into a register
// (lane k holds entry 32 r + k) with the next 32 already in flight, so a request
// never waits on a global load.  Indices must be requested in increasing order.
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

// ------------------------------------------------------------ block compute

// Per-warp constants of the block loop.
template <int NT>
struct WarpConsts {
  uint32_t bq[NT][8][2];  // key-side query fragments
  uint32_t bu[NT][8][2];  // QJL: fragments of S q'
  float inv_qs[NT];       // 1 / query scale of head 4 nt + tig
  float inv_us[NT];
  PTranspose pt;
  uint32_t lk, lv;        // code-table lane bases
  int g_, tig;
};

// Keys of one 16-token block of packed K/V for one warp: base-2 logits u of head
// 4 nt + tig at the lane's tokens g_, g_ + 8 (-inf past ctx or when !valid) and
// their value weights wv (0 when masked), written to u[nt][o], u[nt][o + 1].
template <int NT, int BK, int BV, bool QJL, int T, bool MASKED>
__device__ __forceinline__ void packed_keys(const WarpConsts<NT>& wc, const uint8_t* sk, const uint8_t* sv, int t0,
                                            int ctx, bool valid, float qjl_coef, int o, float (&u)[NT][T],
                                            float (&wv)[T]) {
  constexpr int RK = 16 * BK, RV = 16 * BV;
  const int g_ = wc.g_, tig = wc.tig;
  // ---- keys: 8 k-chunks in KC independent accumulation chains per n-tile (the
  // two blocks of a step give the scheduler a second independent set)
  constexpr int KC = 2;
  float dk[NT][KC][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int p = 0; p < KC; ++p)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[nt][p][e] = 0.0f;
  if constexpr (BK == 8) {
    // FP8 E4M3 keys (k8v4): byte j of a record is coordinate j; word c of the lane's
    // 32 bytes holds coordinates 32 tig + 4c .. 4c + 3, the same k order as the codes
    const uint4* r0 = reinterpret_cast<const uint4*>(sk + g_ * RK + 32 * tig);
    const uint4* r1 = reinterpret_cast<const uint4*>(sk + (g_ + 8) * RK + 32 * tig);
    const uint4 p0 = r0[0], p1 = r0[1], p2 = r1[0], p3 = r1[1];
    const uint32_t kw0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const uint32_t kw1[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t ak[4] = {fp8x2_to_f16x2(kw0[c] & 0xFFFFu), fp8x2_to_f16x2(kw1[c] & 0xFFFFu),
                              fp8x2_to_f16x2(kw0[c] >> 16), fp8x2_to_f16x2(kw1[c] >> 16)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_f16(dk[nt][c % KC], ak, wc.bq[nt][c][0], wc.bq[nt][c][1], dk[nt][c % KC]);
    }
  } else {
    uint32_t kn[2][4];
    load_quarter<BK>(sk + g_ * RK, tig, kn[0]);
    load_quarter<BK>(sk + (g_ + 8) * RK, tig, kn[1]);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int wi = c >> 1, bi = 2 * (c & 1);
      const uint32_t ak[4] = {lut(wc.lk, kn[0][wi], bi), lut(wc.lk, kn[1][wi], bi), lut(wc.lk, kn[0][wi], bi + 1),
                              lut(wc.lk, kn[1][wi], bi + 1)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_f16(dk[nt][c % KC], ak, wc.bq[nt][c][0], wc.bq[nt][c][1], dk[nt][c % KC]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int p = 1; p < KC; ++p)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[nt][0][e] += dk[nt][p][e];
  float sq[NT][2];
  if constexpr (QJL) {  // sign term: rows = tokens, columns = S q' (hi, lo)
    const uint32_t sw0 = *reinterpret_cast<const uint32_t*>(sk + 16 * RK + 64 + 16 * g_ + 4 * tig);
    const uint32_t sw1 = *reinterpret_cast<const uint32_t*>(sk + 16 * RK + 64 + 16 * (g_ + 8) + 4 * tig);
    float dq[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) dq[nt][0] = dq[nt][1] = dq[nt][2] = dq[nt][3] = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      // stored bit 1 = +1: f16x2 of (+-1, +-1) with the sign bits from the complement
      const uint32_t n0 = ~sw0 >> (4 * c), n1 = ~sw1 >> (4 * c);
      const uint32_t a[4] = {0x3C003C00u | ((n0 & 1u) << 15) | ((n0 & 2u) << 30),
                             0x3C003C00u | ((n1 & 1u) << 15) | ((n1 & 2u) << 30),
                             0x3C003C00u | ((n0 & 4u) << 13) | ((n0 & 8u) << 28),
                             0x3C003C00u | ((n1 & 4u) << 13) | ((n1 & 8u) << 28)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16(dq[nt], a, wc.bu[nt][c][0], wc.bu[nt][c][1], dq[nt]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sq[nt][0] = dq[nt][0] + dq[nt][1];
      sq[nt][1] = dq[nt][2] + dq[nt][3];
    }
  }
  const float* gk = reinterpret_cast<const float*>(sk + 16 * RK);
  const float* gv = reinterpret_cast<const float*>(sv + 16 * RV);
  const float gk0 = BK == 8 ? 1.0f : gk[g_], gk1 = BK == 8 ? 1.0f : gk[g_ + 8];  // FP8 keys carry no norm
  const bool in0 = !MASKED || (valid && t0 + g_ < ctx), in1 = !MASKED || (valid && t0 + g_ + 8 < ctx);
  wv[o] = in0 ? gv[g_] : 0.0f;
  wv[o + 1] = in1 ? gv[g_ + 8] : 0.0f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float v0 = gk0 * (dk[nt][0][0] + dk[nt][0][1]) * wc.inv_qs[nt];
    float v1 = gk1 * (dk[nt][0][2] + dk[nt][0][3]) * wc.inv_qs[nt];
    if constexpr (QJL) {
      const float* rh = reinterpret_cast<const float*>(sk + 16 * RK + 64 + 256);
      v0 += qjl_coef * rh[g_] * sq[nt][0] * wc.inv_us[nt];
      v1 += qjl_coef * rh[g_ + 8] * sq[nt][1] * wc.inv_us[nt];
    }
    u[nt][o] = in0 ? v0 : -INFINITY;
    u[nt][o + 1] = in1 ? v1 : -INFINITY;
  }
}

// Values of one block: acc += V_hat^T P' (pk[nt] = P' of the lane's token pair),
// value codes of tokens ta, tb (tile 0) and ta + 8, tb + 8 (tile 1) from stage sv.
template <int NT, int BV>
__device__ __forceinline__ void packed_values(SoftmaxState<NT>& st, const WarpConsts<NT>& wc, const uint8_t* sv,
                                              const uint32_t (&pk)[NT]) {
  constexpr int RV = 16 * BV;
  const int g_ = wc.g_, tig = wc.tig;
  const int ta = tok_a(tig), tb = tok_b(tig);
  uint32_t vw[4][2];
  load_sixteenth<BV>(sv + ta * RV, g_, vw[0]);
  load_sixteenth<BV>(sv + tb * RV, g_, vw[1]);
  load_sixteenth<BV>(sv + (ta + 8) * RV, g_, vw[2]);
  load_sixteenth<BV>(sv + (tb + 8) * RV, g_, vw[3]);
  uint32_t bv[NT][2][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) wc.pt.apply(pk[nt], bv[nt]);
#pragma unroll
  for (int kt = 0; kt < 2; ++kt)
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int wi = mt >> 1, bi = 2 * (mt & 1);
      const uint32_t av[4] = {lut(wc.lv, vw[2 * kt][wi], bi), lut(wc.lv, vw[2 * kt][wi], bi + 1),
                              lut(wc.lv, vw[2 * kt + 1][wi], bi), lut(wc.lv, vw[2 * kt + 1][wi], bi + 1)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16(st.acc[nt][mt], av, bv[nt][kt][0], bv[nt][kt][1], st.acc[nt][mt]);
    }
}

// One 16-token block of raw bf16 K/V for one warp (same fragment layout; bf16
// MMAs, P' split into bf16 hi + lo).
template <int NT>
__device__ __forceinline__ void bf16_block(SoftmaxState<NT>& st, const WarpConsts<NT>& wc, const uint8_t* sk,
                                           const uint8_t* sv, int t0, int ctx) {
  constexpr int RB = kD * 2;  // bytes per token row
  const int g_ = wc.g_, tig = wc.tig;
  const uint4* kr0 = reinterpret_cast<const uint4*>(sk + g_ * RB + 64 * tig);
  const uint4* kr1 = reinterpret_cast<const uint4*>(sk + (g_ + 8) * RB + 64 * tig);
  float dk[NT][2][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[nt][p][e] = 0.0f;
#pragma unroll
  for (int c2 = 0; c2 < 4; ++c2) {
    const uint4 k0 = kr0[c2], k1 = kr1[c2];
    const uint32_t a0[4] = {k0.x, k1.x, k0.y, k1.y};  // chunk 2 c2
    const uint32_t a1[4] = {k0.z, k1.z, k0.w, k1.w};  // chunk 2 c2 + 1
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_bf16(dk[nt][0], a0, wc.bq[nt][2 * c2][0], wc.bq[nt][2 * c2][1], dk[nt][0]);
      mma_bf16(dk[nt][1], a1, wc.bq[nt][2 * c2 + 1][0], wc.bq[nt][2 * c2 + 1][1], dk[nt][1]);
    }
  }
  const bool in0 = t0 + g_ < ctx, in1 = t0 + g_ + 8 < ctx;
  float u[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float v0 = (dk[nt][0][0] + dk[nt][0][1]) + (dk[nt][1][0] + dk[nt][1][1]);
    const float v1 = (dk[nt][0][2] + dk[nt][0][3]) + (dk[nt][1][2] + dk[nt][1][3]);
    u[nt][0] = in0 ? v0 : -INFINITY;
    u[nt][1] = in1 ? v1 : -INFINITY;
  }
  const float ones[2] = {in0 ? 1.0f : 0.0f, in1 ? 1.0f : 0.0f};
  uint32_t pk[NT][1], pl[NT][1];
  softmax_tokens<NT, true, 2>(st, u, ones, pk, pl);
  uint32_t bh[NT][2][2], bl[NT][2][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    wc.pt.apply(pk[nt][0], bh[nt]);
    wc.pt.apply(pl[nt][0], bl[nt]);
  }
#pragma unroll
  for (int kt = 0; kt < 2; ++kt) {
    // coordinates [16 g_, 16 g_ + 16) of tokens ta + 8 kt (F) and tb + 8 kt (S)
    const uint4* rf = reinterpret_cast<const uint4*>(sv + (tok_a(tig) + 8 * kt) * RB + 32 * g_);
    const uint4* rs = reinterpret_cast<const uint4*>(sv + (tok_b(tig) + 8 * kt) * RB + 32 * g_);
    const uint4 f0 = rf[0], f1 = rf[1], s0 = rs[0], s1 = rs[1];
    const uint32_t wf[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    const uint32_t ws[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const uint32_t av[4] = {wf[2 * mt], wf[2 * mt + 1], ws[2 * mt], ws[2 * mt + 1]};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16(st.acc[nt][mt], av, bh[nt][kt][0], bh[nt][kt][1], st.acc[nt][mt]);
        mma_bf16(st.acc[nt][mt], av, bl[nt][kt][0], bl[nt][kt][1], st.acc[nt][mt]);
      }
    }
  }
}

// ------------------------------------------------------------ decode kernel

// Live partial slots.  Chunk ch = unit * splits + s runs on CTA ch / NW; the
// warps of one CTA that share a unit are merged into the slot of the first of
// them, so slot s of a unit is live iff s == 0 or (unit * splits + s) % NW == 0.
__device__ __forceinline__ bool slot_live(int unit, int splits, int s, int nw) {
  return s == 0 || ((int64_t)unit * splits + s) % nw == 0;
}

// KIND 0: packed codes (BK, BV, QJL); KIND 1: bf16 pages.  NT n-tiles of 4 heads
// per warp, NW warps per CTA, one CTA per SM holding all of the SM's shared memory.
// Each warp owns one chunk (a split of one unit's context) and streams its pages
// into its own ring of P stages of SB blocks (K page, V page per block) with
// 16-byte cp.async copies (the load/store path, not the bulk-copy engine: with
// pages of about 1 KB the bulk-copy engine cannot keep enough bytes in flight),
// P - 1 stages ahead of the one it computes on.
// Shared layout (absolute shared addresses; base = start of the dynamic window):
//   packed: rings of warps [0, n_lo) in [base, 0x10000), code tables in
//           [0x10000, 0x20000), rings of the other warps from 0x20000;
//   bf16:   rings from base.  The merge scratch of the epilogue reuses the rings
//   above the tables (drained by then).
template <int KIND, int BK, int BV, bool QJL, int NT>
__host__ __device__ constexpr int decode_stage_blocks() {
  return KIND == 0 ? 2 : 1;
}
template <int KIND, int BK, int BV, bool QJL, int NT>
__host__ __device__ constexpr int decode_ring_stages() {
  return KIND == 1 ? 3 : ((NT == 1 && !QJL) || BK == 8 ? 2 : 3);
}

// Bytes of a K and a V page of the layer formats the decode kernel takes (they
// agree with page_bytes_of; the launcher checks).
template <int KIND, int BK, bool QJL>
__host__ __device__ constexpr int decode_kpage() {
  return KIND == 1 ? kBlock * kD * 2 : (BK == 8 ? kBlock * kD : kBlock * (kD * BK / 8 + 4) + (QJL ? kBlock * (kD / 8 + 4) : 0));
}
template <int KIND, int BV>
__host__ __device__ constexpr int decode_vpage() {
  return KIND == 1 ? kBlock * kD * 2 : kBlock * (kD * BV / 8 + 4);
}

// 16-byte global -> shared copy on the load/store path (cp.async, L2 evict-first).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int KIND, int BK, int BV, bool QJL, int NT, int NW>
__global__ void __launch_bounds__(NW * 32, 1) k_decode(DecodeArgs a) {
  constexpr int HPW = 4 * NT;  // heads per warp
  constexpr int SB = decode_stage_blocks<KIND, BK, BV, QJL, NT>();
  constexpr int PMAX = decode_ring_stages<KIND, BK, BV, QJL, NT>();
  constexpr int KPAGE = decode_kpage<KIND, BK, QJL>(), VPAGE = decode_vpage<KIND, BV>();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_ = lane >> 2, tig = lane & 3;
  constexpr uint32_t blk_bytes = (uint32_t)(KPAGE + VPAGE);
  const uint32_t stage_bytes = SB * blk_bytes;
  const uint32_t base = smem_u32(smem_raw);
  const uint32_t top = (base + (uint32_t)a.smem_bytes) & ~15u;
  const uint32_t lo0 = (base + 127u) & ~127u;
  const uint32_t hi0 = KIND == 0 ? kLutAddr + kLutBytes : lo0;
  // the deepest ring (P <= PMAX stages) of which NW copies fit below and above the tables
  int P = PMAX;
  uint32_t ring_bytes = 0u, n_lo = 0u, n_hi = 0u;
  for (;; --P) {
    ring_bytes = (uint32_t)P * stage_bytes;
    n_lo = (KIND == 0 && kLutAddr > lo0) ? (kLutAddr - lo0) / ring_bytes : 0u;
    n_hi = top > hi0 ? (top - hi0) / ring_bytes : 0u;
    if (n_lo + n_hi >= (uint32_t)NW || P == 1) break;
  }
  const uint32_t red_bytes = (uint32_t)(NW * HPW * kD + 2 * NW * HPW + NW) * 4u;
  const bool layout_ok = (KIND == 1 || (base <= kLutAddr && kLutAddr + kLutBytes <= top)) &&
                         n_lo + n_hi >= (uint32_t)NW && hi0 + red_bytes <= top;
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
  const int head0 = kvh * a.g + hg * HPW;
  const int gc = min(HPW, a.g - hg * HPW);

  // ---- prologue: the long-latency loads first (context length, query rows), then
  // the block ids and the first copies, the code tables while those are in flight
  const int ctx_raw = has ? __ldg(a.ctx_lens + b) : 0;
  // tq_decode_step: the last split's warp usually holds the new token's block, so it
  // requests the new K and V coordinates and the signs now (used below)
  uint2 pf_k = make_uint2(0u, 0u), pf_v = make_uint2(0u, 0u);
  float4 pf_kf = make_float4(0.f, 0.f, 0.f, 0.f), pf_vf = pf_kf, pf_sg = pf_kf;
  const bool pf = KIND == 0 && !QJL && BK <= 4 && a.new_k != nullptr && has && s == a.splits - 1;
  if (pf) {
    const int64_t row = ((int64_t)b * a.Hkv + kvh) * kD + 4 * lane;
    if (a.new_bf16) {
      pf_k = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.new_k) + row));
      pf_v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.new_v) + row));
    } else {
      pf_kf = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.new_k) + row));
      pf_vf = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.new_v) + row));
    }
    pf_sg = make_float4(__ldg(a.rot + 4 * lane), __ldg(a.rot + 4 * lane + 1), __ldg(a.rot + 4 * lane + 2),
                        __ldg(a.rot + 4 * lane + 3));
  }

  // CTA-shared query rotation (q_in_kernel != 0): the rows of this CTA's units are
  // rotated once, one warp per row, into a scratch area past the rings
  const int c0 = blockIdx.x * NW;
  const int c1 = min(c0 + NW, a.chunks);
  const int u0 = c0 / a.splits;
  const int nu = c1 > c0 ? (c1 - 1) / a.splits - u0 + 1 : 0;
  const uint32_t hi_rings = (uint32_t)NW > n_lo ? (uint32_t)NW - n_lo : 0u;
  const uint32_t qs_addr = (hi0 + hi_rings * ring_bytes + 15u) & ~15u;
  const bool q_shared = a.q_in_kernel != 0 && layout_ok && qs_addr + (uint32_t)(nu * HPW * (kD * 4 + 4)) <= top;
  // per row: the key-side MMA fragments of the row's head (512 B, see rotate_row), then
  // after all rows the rows' 1 / scale
  uint32_t* qs = reinterpret_cast<uint32_t*>(gen(qs_addr));
  float* qs_inv = reinterpret_cast<float*>(qs + nu * HPW * kD);
  // raw query coordinates 4 lane .. 4 lane + 3 of rotation row `row` (zeros when absent)
  auto load_rot_row = [&](int row, float (&y)[4]) {
    y[0] = y[1] = y[2] = y[3] = 0.0f;
    const int ur = u0 + row / HPW, h = row % HPW;
    const int ub = ur / per_b, urr = ur - ub * per_b, ukvh = urr / a.ngroups, uhg = urr - ukvh * a.ngroups;
    if (h >= min(HPW, a.g - uhg * HPW)) return;
    const int64_t qrow = (int64_t)ub * a.Hq + ukvh * a.g + uhg * HPW + h;
    if (a.q_bf16) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.q) + qrow * kD) +
                            lane);
      y[0] = __uint_as_float(w.x << 16); y[1] = __uint_as_float(w.x & 0xFFFF0000u);
      y[2] = __uint_as_float(w.y << 16); y[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
      const float4 w = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q) + qrow * kD) + lane);
      y[0] = w.x; y[1] = w.y; y[2] = w.z; y[3] = w.w;
    }
  };
  // q' = H (s * q) / sqrt(d) (or q scaled) of one row into the shared scratch
  auto rotate_row = [&](int row, float (&y)[4]) {
    if (a.q_in_kernel == 1) {  // bits 0, 1 of the coordinate in the lane, bits 2..6 across lanes
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] *= __ldg(a.rot + 4 * lane + k);
      const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
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
    }
    const float f = a.q_in_kernel == 1 ? a.q_scale * 0.08838834764831845f : a.q_scale;
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] *= f;
    // fragments: lane l = 8 t + c holds coordinates 32 t + 4 c + {0..3}, i.e. words
    // (c, j = 0, 1) of quarter t for both parts (fp16 hi and lo with a power-of-two
    // scale per row, or bf16 hi and lo).  Segment (part, t) = 16 words [c][j]; its
    // 16-byte chunk k sits at k ^ ((4 part + t) >> 1) so readers hit distinct banks.
    float scale = 1.0f, inv_scale = 1.0f;
    if (KIND == 0) {
      float mx = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int ebits = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
      scale = ebits > 0 ? pow2i(140 - ebits) : 1.0f;
      inv_scale = ebits > 0 ? pow2i(ebits - 140) : 1.0f;
    }
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float s0 = y[2 * j] * scale, s1 = y[2 * j + 1] * scale;
      float2 back;
      if (KIND == 1) {
        hw[j] = pack_bf162(s0, s1);
        back = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[j]));
        lw[j] = pack_bf162(s0 - back.x, s1 - back.y);
      } else {
        hw[j] = pack_half2(s0, s1);
        back = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
        lw[j] = pack_half2(s0 - back.x, s1 - back.y);
      }
    }
    const int t = lane >> 3, c = lane & 7;
    uint32_t* rowp = qs + row * kD;
    *reinterpret_cast<uint2*>(rowp + 16 * t + 4 * ((c >> 1) ^ (t >> 1)) + 2 * (c & 1)) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(rowp + 16 * (4 + t) + 4 * ((c >> 1) ^ ((4 + t) >> 1)) + 2 * (c & 1)) =
        make_uint2(lw[0], lw[1]);
    if (lane == 0) qs_inv[row] = inv_scale;
  };
  float y0[4];
  const bool row0 = q_shared && warp < nu * HPW;
  if (row0) load_rot_row(warp, y0);  // in flight with the context length

  float qv[NT][32];
  float uv[QJL ? NT : 1][32];
  // this warp's query rows: raw (rotated below) or, after the first copies, the rows the
  // preceding rotation pass wrote
  auto load_q_rows = [&](bool from_pass) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hq = 4 * nt + (g_ >> 1);
      const bool hv = has && hq < gc;
      const int64_t row = (int64_t)b * a.Hq + head0 + (hv ? hq : 0);
      if (!from_pass) {
        load_q_raw(a.q, a.q_bf16 != 0, row, hv, tig, qv[nt]);
      } else {
        load_q(a.qrot + row * kD, hv, tig, qv[nt]);
        if constexpr (QJL) load_q(a.uqjl + row * kD, hv, tig, uv[nt]);
      }
    }
  };
  if (!q_shared && a.q_in_kernel) load_q_rows(false);

  // code tables while the context length, the query rows and the block ids are in
  // flight
  uint4* tab = reinterpret_cast<uint4*>(gen(kLutAddr));
  float cl = 0.0f;  // lane k < 16: key centroid k & MK, lane 16 + k: value centroid k & MV
  if constexpr (KIND == 0) {
    constexpr int MK = (1 << BK) - 1, MV = (1 << BV) - 1;
#pragma unroll
    for (int k = 0; k < 16; ++k) {  // uniform constant loads (a lane-indexed parameter read would serialize)
      if (lane == k) cl = a.cbk.c[k & MK];
      if (lane == 16 + k) cl = a.cbv.c[k & MV];
    }
  }
  // rows [e0, e1) of the tables: row e (pair byte, low nibble first) = f16x2(c[e & 15],
  // c[e >> 4]) once per lane; 16-byte word j of a row holds lanes 4j..4j+3 (j < 8: keys,
  // j >= 8: values)
  auto build_tables = [&](int e0, int e1) {
    if constexpr (KIND == 0) {
      if (layout_ok) {
        for (int i = e0 * 16 + (int)threadIdx.x; i < e1 * 16; i += NW * 32) {
          const int e = i >> 4, vo = (i & 8) ? 16 : 0;
          const float lo = __shfl_sync(0xffffffffu, cl, vo + (e & 15));
          const float hi = __shfl_sync(0xffffffffu, cl, vo + (e >> 4));
          const uint32_t v = pack_half2(lo, hi);
          tab[i] = make_uint4(v, v, v, v);
        }
      }
    }
  };
  // Splits cut the block-table row (max_blocks entries), not the context, so the block
  // ids can be read before the context length arrives; a split past the context is
  // empty.  (The longest sequences set the kernel's length either way.)  Rows much
  // wider than the context are re-split below.
  int j0 = (int)((int64_t)s * a.max_blocks / a.splits);
  int j1r = (int)((int64_t)(s + 1) * a.max_blocks / a.splits);
  BlockIds ids;
  ids.init(a.block_table + (int64_t)b * a.max_blocks + j0, has ? j1r - j0 : 0, lane);
  build_tables(0, 256);

  int ctx = ctx_raw;
  if (ctx < 0 || ctx > a.max_blocks * kBlock) {
    if (lane == 0 && s == 0 && r == 0) flag_status(a.status, TQ_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : a.max_blocks * kBlock;
  }
  const int nblk = (ctx + kBlock - 1) / kBlock;
  // A row much wider than the sequence's context (a table padded to a maximum length)
  // would leave most of the unit's splits past the context and the few others with all
  // of it: split the context instead and read those block ids (warp-uniform).
  if (has && 4 * nblk < 3 * a.max_blocks) {
    j0 = (int)((int64_t)s * nblk / a.splits);
    j1r = (int)((int64_t)(s + 1) * nblk / a.splits);
    ids.init(a.block_table + (int64_t)b * a.max_blocks + j0, j1r - j0, lane);
  }
  const int n_my = has ? max(0, min(j1r, nblk) - j0) : 0;
  const int n_stages = (n_my + SB - 1) / SB;

  // copies of stage k (blocks SB k .. SB k + SB - 1 of the chunk) into slot `slot` of this
  // warp's ring, one cp.async group per stage (an empty group past the end); returns the
  // mask of the blocks copied (a block id out of range is recorded and skipped)
  const uint32_t rw = (uint32_t)warp;
  const uint32_t ring = rw < n_lo ? lo0 + rw * ring_bytes : hi0 + (rw - n_lo) * ring_bytes;
  const uint8_t* kbase = a.kpool + (int64_t)kvh * KPAGE;
  const uint8_t* vbase = a.vpool + (int64_t)kvh * VPAGE;
  const int64_t kstride = (int64_t)a.Hkv * KPAGE, vstride = (int64_t)a.Hkv * VPAGE;
  const uint64_t pol = l2_evict_first_policy();  // pages are read once per call
  auto copy_stage = [&](int k, int slot) -> uint32_t {
    uint32_t m = 0u;
    if (k < n_stages) {
#pragma unroll
      for (int e = 0; e < SB; ++e) {
        const int j = SB * k + e;
        if (j < n_my) {  // warp-uniform
          const int blk = ids.get(j, lane);
          if (blk >= 0 && (int64_t)blk < a.num_blocks) {
            m |= 1u << e;
            // lane copies 16-byte chunks lane, lane + 32, ... of the K page, then of the V page
            const uint32_t d = ring + (uint32_t)slot * stage_bytes + (uint32_t)e * blk_bytes + 16u * (uint32_t)lane;
            const uint8_t* ks = kbase + (int64_t)blk * kstride + 16 * lane;
            const uint8_t* vs = vbase + (int64_t)blk * vstride + 16 * lane;
#pragma unroll
            for (int c = 0; c < KPAGE; c += 512)
              if (c + 512 <= KPAGE || 16 * lane < KPAGE - c) cp_async16(d + (uint32_t)c, ks + c, pol);
#pragma unroll
            for (int c = 0; c < VPAGE; c += 512)
              if (c + 512 <= VPAGE || 16 * lane < VPAGE - c) cp_async16(d + (uint32_t)(KPAGE + c), vs + c, pol);
          } else if (lane == 0) {
            flag_status(a.status, TQ_DEV_BAD_BLOCK);
          }
        }
      }
    }
    cp_async_commit();
    return m;
  };
  // waits until this lane's copies of the oldest stage in flight have landed
  auto wait_oldest = [&]() {
    switch (P) {  // the group count of wait_group is an immediate
      case 6: cp_async_wait<5>(); break;
      case 5: cp_async_wait<4>(); break;
      case 4: cp_async_wait<3>(); break;
      case 3: cp_async_wait<2>(); break;
      case 2: cp_async_wait<1>(); break;
      default: cp_async_wait<0>(); break;
    }
  };

  if (row0) {
    rotate_row(warp, y0);
    for (int row = warp + NW; row < nu * HPW; row += NW) {
      float y[4];
      load_rot_row(row, y);
      rotate_row(row, y);
    }
  }

  // first copies as soon as the block ids are in.  Launched as a programmatic dependent
  // of the append (tq_append_decode): everything above overlaps the append; pages only
  // after it is done.
  uint32_t vm = 0u;  // SB bits per slot: blocks present
  if (a.overlap_append) grid_dep_wait();
  for (int k = 0; k < P; ++k) vm |= copy_stage(k, k) << (SB * k);

  // tq_decode_step: the warp whose chunk holds block (ctx - 1) / 16 quantizes the new K
  // and V vectors of its (sequence, KV head), writes both records to the cache and,
  // once that block's copy has landed, into its own stage (below)
  int fz_stage = -1, fz_e = 0, fz_off = 0;
  uint32_t fz_wk = 0u, fz_wv = 0u;
  float fz_gk = 0.0f, fz_gv = 0.0f;
  if constexpr (KIND == 0 && !QJL && BK <= 4) {
    if (a.new_k != nullptr && has && ctx > 0) {
      const int jl = (ctx - 1) / kBlock;
      if (jl >= j0 && jl < j0 + n_my) {  // warp-uniform
        const int blk = __ldg(a.block_table + (int64_t)b * a.max_blocks + jl);
        const int64_t row = ((int64_t)b * a.Hkv + kvh) * kD + 4 * lane;
        float xk[4], xv[4];
        float4 sg = pf_sg;
        if (!pf) {  // (another split holds the block: load now)
          if (a.new_bf16) {
            pf_k = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.new_k) + row));
            pf_v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.new_v) + row));
          } else {
            pf_kf = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.new_k) + row));
            pf_vf = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.new_v) + row));
          }
          sg = make_float4(__ldg(a.rot + 4 * lane), __ldg(a.rot + 4 * lane + 1), __ldg(a.rot + 4 * lane + 2),
                           __ldg(a.rot + 4 * lane + 3));
        }
        if (a.new_bf16) {
          xk[0] = __uint_as_float(pf_k.x << 16); xk[1] = __uint_as_float(pf_k.x & 0xFFFF0000u);
          xk[2] = __uint_as_float(pf_k.y << 16); xk[3] = __uint_as_float(pf_k.y & 0xFFFF0000u);
          xv[0] = __uint_as_float(pf_v.x << 16); xv[1] = __uint_as_float(pf_v.x & 0xFFFF0000u);
          xv[2] = __uint_as_float(pf_v.y << 16); xv[3] = __uint_as_float(pf_v.y & 0xFFFF0000u);
        } else {
          xk[0] = pf_kf.x; xk[1] = pf_kf.y; xk[2] = pf_kf.z; xk[3] = pf_kf.w;
          xv[0] = pf_vf.x; xv[1] = pf_vf.y; xv[2] = pf_vf.z; xv[3] = pf_vf.w;
        }
        warp_quantize_record<BK>(xk, sg, a.cbk, a.norm_raw != 0, lane, fz_wk, fz_gk);
        warp_quantize_record<BV>(xv, sg, a.cbv, a.norm_raw != 0, lane, fz_wv, fz_gv);
        fz_off = (ctx - 1) % kBlock;
        if (blk >= 0 && (int64_t)blk < a.num_blocks) {  // (an id out of range is flagged by the copy)
          constexpr int RK = 16 * BK, RV = 16 * BV;
          uint8_t* kp = const_cast<uint8_t*>(a.kpool) + ((int64_t)blk * a.Hkv + kvh) * KPAGE;
          uint8_t* vp = const_cast<uint8_t*>(a.vpool) + ((int64_t)blk * a.Hkv + kvh) * VPAGE;
          if (lane < 4 * BK) reinterpret_cast<uint32_t*>(kp + fz_off * RK)[lane] = fz_wk;
          if (lane < 4 * BV) reinterpret_cast<uint32_t*>(vp + fz_off * RV)[lane] = fz_wv;
          if (lane == 0) {
            reinterpret_cast<float*>(kp + 16 * RK)[fz_off] = fz_gk;
            reinterpret_cast<float*>(vp + 16 * RV)[fz_off] = fz_gv;
          }
          fz_stage = (jl - j0) / SB;
          fz_e = (jl - j0) % SB;
        }
      }
    }
  }
  if (!q_shared && !a.q_in_kernel) {  // the pages do not depend on the rotation pass; its rows do
    grid_dep_wait();
    load_q_rows(true);
  }


  // per-warp constants: query fragments of column g_ (head 4 nt + g_ / 2, part g_ & 1)
  WarpConsts<NT> wc;
  wc.g_ = g_;
  wc.tig = tig;
  wc.pt.init(g_, tig);
  wc.lk = kLutAddr | (4u * lane);
  wc.lv = wc.lk + 128u;
  auto q_frags = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (q_shared) {  // fragments and scale prepared by the rotating warp
        const int rbase = (unit - u0) * HPW + 4 * nt;
        const int seg = 4 * (g_ & 1) + tig;
        const uint4* src = reinterpret_cast<const uint4*>(qs + (rbase + (g_ >> 1)) * kD + 16 * seg);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 w = has ? src[k ^ (seg >> 1)] : make_uint4(0u, 0u, 0u, 0u);
          wc.bq[nt][2 * k][0] = w.x;
          wc.bq[nt][2 * k][1] = w.y;
          wc.bq[nt][2 * k + 1][0] = w.z;
          wc.bq[nt][2 * k + 1][1] = w.w;
        }
        wc.inv_qs[nt] = has ? qs_inv[rbase + tig] : 1.0f;  // head 4 nt + tig
        wc.inv_us[nt] = 0.0f;
        continue;
      } else if (a.q_in_kernel == 1) {
        rotate_q_quad(qv[nt], a.rot, tig, a.q_scale);
      } else if (a.q_in_kernel == 2) {
#pragma unroll
        for (int k = 0; k < 32; ++k) qv[nt][k] *= a.q_scale;
      }
      const float iq = make_q_frags<KIND == 1>(qv[nt], g_ & 1, wc.bq[nt]);
      wc.inv_qs[nt] = __shfl_sync(0xffffffffu, iq, 8 * tig);  // scale of head 4 nt + tig
      wc.inv_us[nt] = 0.0f;
      if constexpr (QJL) {
        const float iu = make_q_frags<false>(uv[nt], g_ & 1, wc.bu[nt]);
        wc.inv_us[nt] = __shfl_sync(0xffffffffu, iu, 8 * tig);
      }
    }
  };
  if (!q_shared) q_frags();

  SoftmaxState<NT> st;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    st.M[nt] = -INFINITY;
    st.l[nt] = 0.0f;
    st.R[nt] = 0.0f;
    st.rR[nt] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) st.acc[nt][mt][0] = st.acc[nt][mt][1] = st.acc[nt][mt][2] = st.acc[nt][mt][3] = 0.0f;
  }
  __syncthreads();  // tables (and shared query rows) ready
  if (q_shared) q_frags();

  int slot = 0;
  for (int i = 0; i < n_stages; ++i) {
    wait_oldest();  // this lane's copies of stage i have landed
    __syncwarp();   // ... and every lane's
    const uint32_t m = (vm >> (SB * slot)) & ((1u << SB) - 1u);
    const uint8_t* sa = gen(ring + (uint32_t)slot * stage_bytes);
    if constexpr (KIND == 0 && !QJL && BK <= 4) {
      if (i == fz_stage && ((m >> fz_e) & 1u)) {  // tq_decode_step: the new token into the landed block
        constexpr int RK = 16 * BK, RV = 16 * BV;
        uint8_t* kp = const_cast<uint8_t*>(sa) + fz_e * blk_bytes;
        uint8_t* vp = kp + KPAGE;
        if (lane < 4 * BK) reinterpret_cast<uint32_t*>(kp + fz_off * RK)[lane] = fz_wk;
        if (lane < 4 * BV) reinterpret_cast<uint32_t*>(vp + fz_off * RV)[lane] = fz_wv;
        if (lane == 0) {
          reinterpret_cast<float*>(kp + 16 * RK)[fz_off] = fz_gk;
          reinterpret_cast<float*>(vp + 16 * RV)[fz_off] = fz_gv;
        }
        __syncwarp();
      }
    }
    if constexpr (KIND == 0) {
      if constexpr (SB == 2) {  // two blocks (32 tokens) per stage: keys of both, one softmax update, values of both
        if (m) {
          const uint8_t* sb = sa + blk_bytes;
          const int t0 = (j0 + 2 * i) * kBlock;
          float u[NT][4], wv[4];
          if (m == 3u && t0 + 2 * kBlock <= ctx) {  // both blocks whole: no masks
            packed_keys<NT, BK, BV, QJL, 4, false>(wc, sa, sa + KPAGE, t0, ctx, true, a.qjl_coef, 0, u, wv);
            packed_keys<NT, BK, BV, QJL, 4, false>(wc, sb, sb + KPAGE, t0 + kBlock, ctx, true, a.qjl_coef, 2, u, wv);
          } else {
            packed_keys<NT, BK, BV, QJL, 4, true>(wc, sa, sa + KPAGE, t0, ctx, (m & 1u) != 0, a.qjl_coef, 0, u, wv);
            packed_keys<NT, BK, BV, QJL, 4, true>(wc, sb, sb + KPAGE, t0 + kBlock, ctx, (m & 2u) != 0, a.qjl_coef,
                                                  2, u, wv);
          }
          uint32_t pk[NT][2], pl[NT][2];
          softmax_tokens<NT, false, 4>(st, u, wv, pk, pl);
          uint32_t pka[NT], pkb[NT];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            pka[nt] = pk[nt][0];
            pkb[nt] = pk[nt][1];
          }
          packed_values<NT, BV>(st, wc, sa + KPAGE, pka);
          packed_values<NT, BV>(st, wc, sb + KPAGE, pkb);
        }
      } else {  // one block (16 tokens) per stage
        if (m) {
          const int t0 = (j0 + i) * kBlock;
          float u[NT][2], wv[2];
          if (t0 + kBlock <= ctx) {
            packed_keys<NT, BK, BV, QJL, 2, false>(wc, sa, sa + KPAGE, t0, ctx, true, a.qjl_coef, 0, u, wv);
          } else {
            packed_keys<NT, BK, BV, QJL, 2, true>(wc, sa, sa + KPAGE, t0, ctx, true, a.qjl_coef, 0, u, wv);
          }
          uint32_t pk[NT][1], pl[NT][1];
          softmax_tokens<NT, false, 2>(st, u, wv, pk, pl);
          uint32_t pka[NT];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) pka[nt] = pk[nt][0];
          packed_values<NT, BV>(st, wc, sa + KPAGE, pka);
        }
      }
    } else {
      if (m) bf16_block<NT>(st, wc, sa, sa + KPAGE, (j0 + i) * kBlock, ctx);
    }
    __syncwarp();  // every lane is done with the slot
    vm = (vm & ~(((1u << SB) - 1u) << (SB * slot))) | (copy_stage(i + P, slot) << (SB * slot));
    if (++slot == P) slot = 0;
  }
  cp_async_wait<0>();  // (only empty groups remain)

  // ---- epilogue 1: per-warp results to shared memory (true sums, l over the head's lanes)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    st.l[nt] = col_sum(st.l[nt]);
    const float rs = st.R[nt] * (1.0f / kPScale);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.acc[nt][mt][e] *= rs;
  }
  __syncthreads();  // every ring is drained: reuse the stage memory
  float* racc = reinterpret_cast<float*>(gen(hi0));  // [NW warps][HPW heads][128]
  float* rm = racc + NW * HPW * kD;                   // [NW][HPW]
  float* rl = rm + NW * HPW;                          // [NW][HPW]
  int* last_flag = reinterpret_cast<int*>(rl + NW * HPW);  // [NW] units this CTA completes
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hl = 4 * nt + tig;
    float4* dst = reinterpret_cast<float4*>(racc + (warp * HPW + hl) * kD + 16 * g_);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
      dst[mt] = make_float4(st.acc[nt][mt][0], st.acc[nt][mt][1], st.acc[nt][mt][2], st.acc[nt][mt][3]);
    if (g_ == 0) {
      rm[warp * HPW + hl] = st.M[nt];
      rl[warp * HPW + hl] = st.l[nt];
    }
  }
  __syncthreads();

  // ---- epilogue 2: one partial per (unit present in this CTA, head), all threads
  if (!layout_ok || c0 >= c1) return;  // uniform
  for (int it = threadIdx.x; it < nu * HPW * 32; it += NW * 32) {
    const int ui = it / (HPW * 32), h = (it >> 5) % HPW, qd = it & 31;
    const int u = u0 + ui;
    const int ub = u / per_b, ur = u - ub * per_b, ukvh = ur / a.ngroups, uhg = ur - ukvh * a.ngroups;
    if (h >= min(HPW, a.g - uhg * HPW)) continue;
    const int wb = max(u * a.splits, c0) - c0, we = min((u + 1) * a.splits, c1) - c0;
    float M = -INFINITY;
    for (int w = wb; w < we; ++w) M = fmaxf(M, rm[w * HPW + h]);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float L = 0.0f;
    for (int w = wb; w < we; ++w) {
      const float mw = rm[w * HPW + h];
      const float f = (mw == -INFINITY) ? 0.0f : pow2i((int)(mw - M));  // maxima are integral
      const float4 v = *reinterpret_cast<const float4*>(racc + (w * HPW + h) * kD + 4 * qd);
      acc.x = fmaf(v.x, f, acc.x);
      acc.y = fmaf(v.y, f, acc.y);
      acc.z = fmaf(v.z, f, acc.z);
      acc.w = fmaf(v.w, f, acc.w);
      L = fmaf(rl[w * HPW + h], f, L);
    }
    const int slot = c0 + wb - u * a.splits;
    const int64_t row = ((int64_t)ub * a.Hq + ukvh * a.g + uhg * HPW + h) * a.splits + slot;
    *reinterpret_cast<float4*>(a.part + row * kD + 4 * qd) = acc;
    if (qd == 0) {
      a.ml[row * 2] = M;
      a.ml[row * 2 + 1] = L;
    }
  }
  if (!a.fuse_combine) return;

  // ---- epilogue 3: the CTA that completes a unit merges its slots and applies Pi^T.
  // The partials of all threads are ordered before the count by the barrier and one
  // release per unit; the completing CTA acquires the count before the barrier that
  // lets its threads read the other CTAs' partials.
  __syncthreads();
  if (threadIdx.x < nu) {
    grid_dep_wait();  // the counters may be zeroed by a preceding pass
    const int u = u0 + threadIdx.x;
    const int covered = min((u + 1) * a.splits, c1) - max(u * a.splits, c0);
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(a.counters + u), "r"(covered) : "memory");
    const bool last = old + covered == a.splits;
    if (last) a.counters[u] = 0;  // every chunk of the unit has counted: ready for the next call
    last_flag[threadIdx.x] = last ? 1 : 0;
  }
  __syncthreads();
  // a dense Pi for the inverse rotation: staged row-major in the code-table region (free
  // now) when this CTA completes a unit; lanes then read distinct banks of one row
  const float* pim = reinterpret_cast<const float*>(gen(kLutAddr));
  if constexpr (KIND == 0) {
    if (a.fuse_combine == 3) {
      bool any = false;
      for (int ui = 0; ui < nu; ++ui) any |= last_flag[ui] != 0;
      if (any) {  // uniform; a thread's loads go out four at a time
        constexpr int kIters = (kD * kD / 4 + NW * 32 - 1) / (NW * 32);
#pragma unroll
        for (int i0 = 0; i0 < kIters; i0 += 4) {
          float4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = (int)threadIdx.x + (i0 + i) * NW * 32;
            if (i0 + i < kIters && e < kD * kD / 4) v[i] = __ldg(reinterpret_cast<const float4*>(a.rot) + e);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = (int)threadIdx.x + (i0 + i) * NW * 32;
            if (i0 + i < kIters && e < kD * kD / 4) reinterpret_cast<float4*>(gen(kLutAddr))[e] = v[i];
          }
        }
        __syncthreads();
      }
    }
  }
  // one warp per (completed unit, head) row; lane holds coordinates 4 lane .. 4 lane + 3:
  // merge the unit's live slots, divide by the denominator, apply Pi^T in registers
  for (int rr = warp; rr < nu * HPW; rr += NW) {
    const int ui = rr / HPW, h = rr - (rr / HPW) * HPW;
    if (!last_flag[ui]) continue;  // warp-uniform
    const int u = u0 + ui;
    const int ub = u / per_b, ur = u - ub * per_b, ukvh = ur / a.ngroups, uhg = ur - ukvh * a.ngroups;
    if (h >= min(HPW, a.g - uhg * HPW)) continue;
    const int64_t hrow = (int64_t)ub * a.Hq + ukvh * a.g + uhg * HPW + h;
    // live slots: 0, then f1, f1 + NW, ... (the first chunk of the unit on each later CTA)
    const int f1 = NW - (int)(((int64_t)u * a.splits) % NW);
    float m4[4], l4[4];
    float4 v4[4];
    // the signs of the inverse FWHT, loaded with the slots
    float4 sgn = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (a.fuse_combine == 2) {
      if ((reinterpret_cast<uintptr_t>(a.rot) & 15u) == 0u) {
        sgn = __ldg(reinterpret_cast<const float4*>(a.rot) + lane);
      } else {
        sgn = make_float4(__ldg(a.rot + 4 * lane), __ldg(a.rot + 4 * lane + 1), __ldg(a.rot + 4 * lane + 2),
                          __ldg(a.rot + 4 * lane + 3));
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // the loads of up to four slots in flight together
      const int s2 = k == 0 ? 0 : f1 + (k - 1) * NW;
      const int64_t row = hrow * a.splits + s2;
      const bool in = s2 < a.splits;
      m4[k] = in ? __ldcg(a.ml + row * 2) : -INFINITY;
      l4[k] = in ? __ldcg(a.ml + row * 2 + 1) : 0.0f;
      v4[k] = in ? __ldcg(reinterpret_cast<const float4*>(a.part + row * kD) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float M = -INFINITY, L = 0.0f;
    auto merge = [&](float m, float l, const float4& v) {
      if (m == -INFINITY) return;
      const float nm = fmaxf(M, m);
      const float fo = (M == -INFINITY) ? 0.0f : pow2i((int)(M - nm)), fn = pow2i((int)(m - nm));
      y[0] = y[0] * fo + v.x * fn;
      y[1] = y[1] * fo + v.y * fn;
      y[2] = y[2] * fo + v.z * fn;
      y[3] = y[3] * fo + v.w * fn;
      L = L * fo + l * fn;
      M = nm;
    };
#pragma unroll
    for (int k = 0; k < 4; ++k) merge(m4[k], l4[k], v4[k]);
    for (int s2 = f1 + 3 * NW; s2 < a.splits; s2 += NW) {  // more than four slots
      const int64_t row = hrow * a.splits + s2;
      merge(__ldcg(a.ml + row * 2), __ldcg(a.ml + row * 2 + 1),
            __ldcg(reinterpret_cast<const float4*>(a.part + row * kD) + lane));
    }
    const float inv_l = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] *= inv_l;
    if (a.fuse_combine == 2) {  // Pi^T y = D H y / sqrt(d): bits 0, 1 in the lane, bits 2..6 across lanes
      const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
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
      y[0] *= 0.08838834764831845f * sgn.x;
      y[1] *= 0.08838834764831845f * sgn.y;
      y[2] *= 0.08838834764831845f * sgn.z;
      y[3] *= 0.08838834764831845f * sgn.w;
    } else if (a.fuse_combine == 3) {  // Pi^T y for a dense Pi: (Pi^T y)_c = sum_j Pi[j][c] y_j
      float o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int j4 = 0; j4 < 32; ++j4) {
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float yj = __shfl_sync(0xffffffffu, y[k2], j4);  // y_j, j = 4 j4 + k2
          const float4 p = reinterpret_cast<const float4*>(pim + (4 * j4 + k2) * kD)[lane];
          o[0] = fmaf(p.x, yj, o[0]);
          o[1] = fmaf(p.y, yj, o[1]);
          o[2] = fmaf(p.z, yj, o[2]);
          o[3] = fmaf(p.w, yj, o[3]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = o[k];
    }
    const int64_t orow = hrow * kD + 4 * lane;
    if (a.out_bf16) {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.out) + orow;
      if ((reinterpret_cast<uintptr_t>(a.out) & 7u) == 0u) {  // one 8-byte store
        *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf162(y[0], y[1]), pack_bf162(y[2], y[3]));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = __float2bfloat16_rn(y[k]);
      }
    } else {
      float* o = reinterpret_cast<float*>(a.out) + orow;
      if ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0u) {  // one 16-byte store
        *reinterpret_cast<float4*>(o) = make_float4(y[0], y[1], y[2], y[3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = y[k];
      }
    }
  }
}

// ------------------------------------------------------------- prologue

enum { ROTQ_IDENTITY = 0, ROTQ_HADAMARD = 1, ROTQ_DENSE = 2 };

// One warp per (sequence, query head), 16 per CTA.  qrot = Pi q * scale; uq = S qrot
// (QJL).  Also zeroes the decode's per-unit chunk counters.  The decode kernel that
// follows is launched as its programmatic dependent: it may start right away and waits
// for this grid (griddepcontrol.wait) only where it reads qrot / uq or the counters.
// A dense Pi and S are staged once per CTA in shared memory, M[c][j] at row c, column
// j ^ (c & 31), so that lane l forming outputs l + 32 k reads 32 distinct banks.
constexpr int kRotWarps = 16;

// out[k] = (M x)_{lane + 32 k} from the staged M; x_j is held by lane j >> 2 at x4[j & 3]
// (4-per-lane layout) when four_per_lane, else by lane j & 31 at x4[j >> 5].
__device__ __forceinline__ void staged_matvec(const float* M, const float (&x4)[4], bool four_per_lane, int lane,
                                              float (&out)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) out[k] = 0.0f;
#pragma unroll 4
  for (int j = 0; j < kD; ++j) {
    const float xj = four_per_lane ? __shfl_sync(0xffffffffu, j & 1 ? (j & 2 ? x4[3] : x4[1]) : (j & 2 ? x4[2] : x4[0]), j >> 2)
                                   : __shfl_sync(0xffffffffu, j & 64 ? (j & 32 ? x4[3] : x4[2]) : (j & 32 ? x4[1] : x4[0]),
                                                 j & 31);
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = fmaf(M[(lane + 32 * k) * kD + (j ^ lane)], xj, out[k]);
  }
}

// (a CTA of kRotWarps warps; each thread's loads are all in flight before its stores)
__device__ __forceinline__ void stage_swizzled(const float* __restrict__ src, float* M) {
  constexpr int kThreads = kRotWarps * 32, kIters = kD * kD / 4 / kThreads;
  static_assert(kIters * kThreads == kD * kD / 4, "whole float4 per thread");
  float4 v[kIters];
#pragma unroll
  for (int i = 0; i < kIters; ++i) v[i] = __ldg(reinterpret_cast<const float4*>(src) + threadIdx.x + i * kThreads);
#pragma unroll
  for (int i = 0; i < kIters; ++i) {  // float4 e of row c = e / 32
    const int e = threadIdx.x + i * kThreads;
    const int c = e >> 5, j = 4 * (e & 31);
    float* row = M + c * kD;
    const int sw = c & 31;
    row[(j + 0) ^ sw] = v[i].x;
    row[(j + 1) ^ sw] = v[i].y;
    row[(j + 2) ^ sw] = v[i].z;
    row[(j + 3) ^ sw] = v[i].w;
  }
}

template <typename TQ>
__global__ void __launch_bounds__(kRotWarps * 32) k_rotate_q(const TQ* __restrict__ q, int64_t n_rows, int kind,
                                                             const float* __restrict__ rot,
                                                             const float* __restrict__ S, float scale, float* qrot,
                                                             float* uq, int* counters, int n_counters) {
  extern __shared__ __align__(16) float mat[];  // [128][128] staged Pi or S (dense and QJL only)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_counters; i += gridDim.x * blockDim.x) counters[i] = 0;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRotWarps + (threadIdx.x >> 5);
  const bool live = row < n_rows;
  const TQ* src = q + (live ? row : 0) * kD;
  float x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = live ? load_elem<TQ>(src + 4 * lane + k) : 0.0f;
  float y[4];
  bool y_strided = false;  // y in the lane + 32 k layout (else coordinates 4 lane .. 4 lane + 3)
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
    stage_swizzled(rot, mat);
    __syncthreads();
    staged_matvec(mat, x, true, lane, y);
    y_strided = true;
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] *= scale;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = x[k] * scale;
  }
  if (live) {
    if (y_strided) {
#pragma unroll
      for (int k = 0; k < 4; ++k) qrot[row * kD + lane + 32 * k] = y[k];
    } else {
      *reinterpret_cast<float4*>(qrot + row * kD + 4 * lane) = make_float4(y[0], y[1], y[2], y[3]);
    }
  }
  if (S) {
    if (kind == ROTQ_DENSE) __syncthreads();  // every warp is done with the staged Pi
    stage_swizzled(S, mat);
    __syncthreads();
    float z[4];
    staged_matvec(mat, y, !y_strided, lane, z);
    if (live) {
#pragma unroll
      for (int k = 0; k < 4; ++k) uq[row * kD + lane + 32 * k] = z[k];
    }
  }
  // Launched as a programmatic dependent of the append (tq_append_decode), this pass
  // touches none of the append's memory but completes only after it, so the decode that
  // waits for this pass finds the pages written.  (No-op for an ordinary launch.)
  grid_dep_wait();
}

// ------------------------------------------------------------- combine

// Heads of a decode unit and the CTA width of the decode launch, for the live slots.
struct UnitMap {
  int Hq, Hkv, g, hpw, ngroups, nw;
};

template <typename TO>
__global__ void __launch_bounds__(128) k_combine(const float* __restrict__ part, const float* __restrict__ ml,
                                                 int splits, UnitMap um, int kind, const float* __restrict__ rot,
                                                 TO* out) {
  __shared__ float sm[256], sl[256], y[kD];
  __shared__ float stot[4];
  const int t = threadIdx.x;
  const int64_t bh = blockIdx.x;
  const int bq = (int)(bh / um.Hq), head = (int)(bh - (int64_t)bq * um.Hq);
  const int unit = (bq * um.Hkv + head / um.g) * um.ngroups + (head % um.g) / um.hpw;
  float mx = -INFINITY;
  for (int s = t; s < splits; s += blockDim.x)
    if (slot_live(unit, splits, s, um.nw)) mx = fmaxf(mx, ml[(bh * splits + s) * 2]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) stot[t >> 5] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(stot[0], stot[1]), fmaxf(stot[2], stot[3]));
  for (int s = t; s < splits; s += blockDim.x) {
    const float ms = slot_live(unit, splits, s, um.nw) ? ml[(bh * splits + s) * 2] : -INFINITY;
    const float f = (ms == -INFINITY) ? 0.0f : pow2i((int)(ms - M));  // maxima are integral
    sm[s] = f;
    sl[s] = f > 0.0f ? ml[(bh * splits + s) * 2 + 1] * f : 0.0f;
  }
  __syncthreads();
  float acc = 0.0f, L = 0.0f;
  for (int s = 0; s < splits; ++s) {
    if (sm[s] == 0.0f) continue;  // empty chunk or merged into another slot
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

// Warps per decode CTA (one CTA per SM): 16 for packed pages with groups of <= 4
// query heads, 12 for groups of 8 and for FP8 keys (larger stages), 8 for QJL keys
// and bf16 pages (more registers).
constexpr int decode_nw(bool packed_plain, int nt, bool fp8_keys = false, bool qjl = false) {
  // QJL keys with groups of <= 4 heads fit 16 warps' registers (128 each, rings of two
  // stages); with groups of 8, and for bf16 pages, 8 warps
  return packed_plain ? ((nt == 1 && !fp8_keys) ? 16 : 12) : ((qjl && nt == 1) ? 16 : 8);
}

int decode_warps(const tq_cache_desc& d, int g) {
  if (d.fmt.kv_format == TQ_KV_POLAR) return g <= 4 ? 12 : 8;  // three (two) CTAs of four warps per SM
  const bool k8 = d.fmt.kv_format == TQ_KV_K8V4;
  const bool qjl = d.fmt.kv_format == TQ_KV_PACKED && d.fmt.qjl_k;
  return decode_nw((d.fmt.kv_format == TQ_KV_PACKED && !d.fmt.qjl_k) || k8, g <= 4 ? 1 : 2, k8, qjl);
}

template <int KIND, int BK, int BV, bool QJL, int NT>
static cudaError_t run_decode_nt(DecodeArgs a, cudaStream_t st) {
  constexpr int NW = decode_nw(KIND == 0 && !QJL, NT, BK == 8, QJL);
  if (a.kpage != decode_kpage<KIND, BK, QJL>() || a.vpage != decode_vpage<KIND, BV>()) return cudaErrorInvalidValue;
  auto kern = k_decode<KIND, BK, BV, QJL, NT, NW>;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  a.smem_bytes = optin;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  // programmatic dependent of the rotation / counter pass when one was launched just before
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.chunks + NW - 1) / NW));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = (size_t)optin;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;  // otherwise the previous kernel may be anything that writes the inputs
  e = cudaLaunchKernelEx(&cfg, kern, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Heads per warp: 4 (one n-tile) for GQA groups of up to 4 query heads, else 8.
template <int KIND, int BK, int BV, bool QJL>
static cudaError_t run_decode(const DecodeArgs& a, cudaStream_t st) {
  return a.g <= 4 ? run_decode_nt<KIND, BK, BV, QJL, 1>(a, st) : run_decode_nt<KIND, BK, BV, QJL, 2>(a, st);
}

template <int BK, bool QJL>
static cudaError_t dispatch_bv(const DecodeArgs& a, int bv, cudaStream_t st) {
  switch (bv) {
    case 2: return run_decode<0, BK, 2, QJL>(a, st);
    case 3: return run_decode<0, BK, 3, QJL>(a, st);
    default: return run_decode<0, BK, 4, QJL>(a, st);
  }
}

cudaError_t launch_decode(const DecodeCall& c, cudaStream_t st) {
  const tq_cache_desc& d = *c.desc;
  if (d.fmt.kv_format == TQ_KV_POLAR) return launch_polar_decode(c, st);
  const bool bf16 = d.fmt.kv_format == TQ_KV_BF16;
  const bool k8 = d.fmt.kv_format == TQ_KV_K8V4;  // FP8 keys (unrotated) with packed values
  const bool qjl = !bf16 && !k8 && d.fmt.qjl_k;
  const DecodeWorkspace ws = decode_workspace(c.batch, c.num_q_heads, c.splits, kD, qjl);
  float* qrot = reinterpret_cast<float*>(c.workspace + ws.qrot_off);
  float* uq = qjl ? qrot + (size_t)c.batch * c.num_q_heads * kD : nullptr;
  // the output's inverse rotation is the values' rotation; the query is rotated like the
  // keys, i.e. not at all for bf16 and FP8 keys
  const int kind = bf16 ? ROTQ_IDENTITY : (d.fmt.rot_kind == TQ_ROT_DENSE ? ROTQ_DENSE : ROTQ_HADAMARD);
  const int kind_q = k8 ? ROTQ_IDENTITY : kind;
  const int64_t rows = (int64_t)c.batch * c.num_q_heads;
  const float scale = c.sm_scale * kLog2e;
  int* counters = reinterpret_cast<int*>(c.workspace + ws.cnt_off);
  // Hadamard and unrotated layers without QJL rotate q inside the decode kernel;
  // dense rotations and S q' (QJL) take a separate mat-vec pass first
  const bool q_aligned = (reinterpret_cast<uintptr_t>(c.q) & 15) == 0;
  const int q_in_kernel = (!qjl && kind_q != ROTQ_DENSE && q_aligned) ? (kind_q == ROTQ_HADAMARD ? 1 : 2) : 0;
  // The chunk counters stay zero between calls (the decode kernel resets each unit's
  // counter when it completes the unit), so the separate pass is needed only for a
  // q mat-vec or for counters that do not fit the fixed region at the start of the
  // workspace (its contents must be zero before the first call).
  const int g = c.num_q_heads / d.num_kv_heads;
  const int64_t units = (int64_t)c.batch * d.num_kv_heads * ((g + (g <= 4 ? 3 : 7)) / (g <= 4 ? 4 : 8));
  const bool prep = !q_in_kernel || (size_t)units * sizeof(int32_t) > kCounterRegionBytes;
  if (prep) {
    const int64_t rot_rows = q_in_kernel ? 0 : rows;
    const int n_counters = (int)rows;  // >= batch * kv heads * head groups
    unsigned rgrid = (unsigned)((rot_rows + kRotWarps - 1) / kRotWarps);
    if (rgrid == 0) rgrid = (unsigned)((n_counters + kRotWarps * 32 - 1) / (kRotWarps * 32));
    const bool staged = rot_rows > 0 && (kind_q == ROTQ_DENSE || qjl);
    const size_t smem = staged ? (size_t)kD * kD * sizeof(float) : 0;
    // after this library's append (tq_append_decode) the pass is its programmatic
    // dependent: it reads only q and writes only the workspace, so it overlaps the append
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rgrid);
    cfg.blockDim = dim3(kRotWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.after_append ? 1 : 0;
    const float* S = qjl ? d.qjl_proj : nullptr;
    cudaError_t ea = cudaSuccess;
    if (c.q_dtype == TQ_F32) {
      if (staged) ea = cudaFuncSetAttribute(k_rotate_q<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (ea == cudaSuccess)
        ea = cudaLaunchKernelEx(&cfg, k_rotate_q<float>, reinterpret_cast<const float*>(c.q), rot_rows, kind_q,
                                (const float*)d.rotation, S, scale, qrot, uq, counters, n_counters);
    } else {
      if (staged)
        ea = cudaFuncSetAttribute(k_rotate_q<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (ea == cudaSuccess)
        ea = cudaLaunchKernelEx(&cfg, k_rotate_q<__nv_bfloat16>, reinterpret_cast<const __nv_bfloat16*>(c.q),
                                rot_rows, kind_q, (const float*)d.rotation, S, scale, qrot, uq, counters, n_counters);
    }
    if (ea != cudaSuccess) return ea;
    count_launch();
  }
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
  a.q = c.q;
  a.q_bf16 = c.q_dtype == TQ_BF16 ? 1 : 0;
  a.q_in_kernel = q_in_kernel;
  a.q_scale = scale;
  // programmatic dependent of the prep pass, or of the append of tq_append_decode (the
  // prep pass itself is an ordinary launch, so it starts after the append has finished)
  a.pdl = (prep || c.after_append) ? 1 : 0;
  // after the append: wait before the first page copy (with a query pass in between, the
  // pass completes only after the append)
  a.overlap_append = c.after_append ? 1 : 0;
  a.Hq = c.num_q_heads;
  a.g = c.num_q_heads / d.num_kv_heads;
  a.ngroups = (a.g + (a.g <= 4 ? 3 : 7)) / (a.g <= 4 ? 4 : 8);  // head groups of 4 or 8 per warp
  a.splits = c.splits;
  a.chunks = c.batch * d.num_kv_heads * a.ngroups * c.splits;
  a.part = reinterpret_cast<float*>(c.workspace + ws.part_off);
  a.ml = reinterpret_cast<float*>(c.workspace + ws.ml_off);
  a.cbk = codebook_of(d, 0);
  a.cbv = codebook_of(d, 1);
  a.qjl_coef = 1.2533141373155003f / (float)kD;  // sqrt(pi/2) / m
  a.status = c.status;
  // the decode kernel finishes the job itself (merge and inverse rotation) unless the
  // splits are too many for its merge or the dense rotation's rows are not 16-byte aligned
  const bool rot_aligned = (reinterpret_cast<uintptr_t>(d.rotation) & 15) == 0;
  a.fuse_combine = (c.splits > kMaxFusedSplits || (kind == ROTQ_DENSE && !rot_aligned))
                       ? 0
                       : (kind == ROTQ_HADAMARD ? 2 : (kind == ROTQ_DENSE ? 3 : 1));
  a.counters = counters;
  a.rot = d.rotation;
  a.out = c.out;
  a.out_bf16 = c.out_dtype == TQ_BF16 ? 1 : 0;
  a.new_k = c.new_k;
  a.new_v = c.new_v;
  a.new_bf16 = c.new_dtype == TQ_BF16 ? 1 : 0;
  a.norm_raw = d.fmt.norm_mode == TQ_NORM_RAW ? 1 : 0;
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
        case 8: e = dispatch_bv<8, false>(a, bv, st); break;  // FP8 keys (k8v4)
        default: e = dispatch_bv<4, false>(a, bv, st); break;
      }
    }
  }
  if (e != cudaSuccess) return e;
  if (a.fuse_combine) return cudaSuccess;
  const unsigned cgrid = (unsigned)rows;
  UnitMap um;
  um.Hq = a.Hq;
  um.Hkv = a.Hkv;
  um.g = a.g;
  um.hpw = a.g <= 4 ? 4 : 8;
  um.ngroups = a.ngroups;
  um.nw = decode_warps(d, a.g);
  if (c.out_dtype == TQ_F32)
    k_combine<float><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, um, kind, d.rotation,
                                            reinterpret_cast<float*>(c.out));
  else
    k_combine<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, um, kind, d.rotation,
                                                    reinterpret_cast<__nv_bfloat16*>(c.out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace tq
