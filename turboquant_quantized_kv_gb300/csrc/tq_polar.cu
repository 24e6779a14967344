// PolarQuant-variant layers of libtq (sm_103a): append, dequantize, decode.
//
// What is computed (lilting.ch TurboQuant article, "PolarQuant: 極座標変換で量子化
// 定数を不要にする"): the Hadamard-rotated vector y = Pi x is turned into polar
// form recursively -- coordinate pairs give radii and angles, radii are paired
// again -- down to one radius and d - 1 angles; each angle is coded on a fixed
// uniform grid (b bits, no per-block constants) and the radius is kept as fp16.
// Grids and the record layout are specified in include/tq.h.
//
// Angle codes without trigonometry.  With squared radii s = rho^2 of a pair
// (a, b) >= 0, theta >= e  <=>  b^2 >= a^2 tan^2(e) for e in [0, pi/2), so a
// level-l (l >= 2) code is the number of grid edges e_k = k pi / 2^(b+1) with
// s_b >= s_a tan^2(e_k): with u = min / max of the two squared radii, a 256-cell
// table over u gives the count below pi/4 up to one more edge test, mirrored
// above pi/4.  Level 1 (the whole circle) takes the quadrant of
// (-y_{2i}, -y_{2i+1}) -- phi = theta + pi mod 2 pi -- from the signs, then one
// exact (pi/4) and one tan^2 test inside the quadrant.  Only squared sums are
// carried up the levels: no sqrt, no atan2.
//
// Kernels:
//   k_polar_append   4 lanes per vector (lane q holds y[32q, 32q + 32)): signs on
//                    the packed bf16 words, packed-pair FWHT, 31 angles per lane,
//                    the last two levels from the quad's four squared radii;
//                    codes are staged per vector in shared memory so lane q packs
//                    and writes record bits [32 b q, 32 b (q + 1)).
//   k_polar_decode   (tq_polar.cuh) one warp per (sequence, KV head, head group,
//                    split) chunk; pages stream through a two-stage cp.async ring
//                    of two blocks (32 tokens: lane = token).  Key logits in fp32
//                    pairs from the depth-first rebuild of each key's unit
//                    direction; value directions through an fp16 tile into
//                    tensor-core MMAs.  One partial per (query head, split).
//   k_polar_combine  CTA per (sequence, query head): log-sum-exp merge of the
//                    splits and the inverse rotation Pi^T.
//   k_polar_dequant  warp per 32 vectors: x_hat = r Pi^T y_hat.
#include "tq_polar.cuh"

namespace tq {
static PolarGrid polar_grid(int bits) {
  PolarGrid g = {};
  const int n = 1 << bits, m = n / 4;
  const double pi = 3.14159265358979323846;
  const double w1 = 2.0 * pi / n, wh = 0.5 * pi / n;
  for (int k = 1; k < m; ++k) {
    const double t = std::tan(k * w1);
    g.t1[k] = (float)(t * t);
  }
  for (int k = 1; k < n; ++k) {
    const double t = std::tan(k * wh);
    g.th[k] = (float)(t * t);
  }
  // cell table over u = min / max of a pair's squared radii in [0, 1]: the edges with
  // tan^2 <= 1 are at least 0.0097 apart (4 bits), so no cell of 1/256 holds two
  for (int i = 0; i < 256; ++i) {
    int c = 0;
    for (int k = 1; k < n; ++k) c += (double)g.th[k] <= i / 256.0 ? 1 : 0;
    g.ucell[i] = (uint8_t)c;
  }
  for (int k = 0; k < n; ++k) {
    const double a1 = (k + 0.5) * w1 - pi, ah = (k + 0.5) * wh;
    g.cs1[2 * k] = (float)std::cos(a1);
    g.cs1[2 * k + 1] = (float)std::sin(a1);
    g.csh[2 * k] = (float)std::cos(ah);
    g.csh[2 * k + 1] = (float)std::sin(ah);
  }
  return g;
}

// Code of a level >= 2 angle from the squared radii (sa, sb) of its pair:
// #{k : sb >= sa tan^2(e_k)}.  With u = min / max in [0, 1] the count below pi/4 is
// ucell[floor(256 u)] plus one more if u passes the next edge; above pi/4
// (sb > sa) the angle is pi/2 - atan(sqrt u) and the count is mirrored.  A pair of
// two zeros has angle 0 (u = 0, no mirror).
template <int BITS>
__device__ __forceinline__ uint32_t code_high(float sa, float sb, const float* th, const uint8_t* ucell) {
  constexpr uint32_t N = 1u << BITS;
  const bool up = sb > sa;
  const float lo = up ? sa : sb, hi = up ? sb : sa;
  const float u = hi > 0.0f ? __fdividef(lo, hi) : 0.0f;
  const uint32_t k0 = ucell[min((int)(u * 256.0f), 255)];
  const uint32_t c = k0 + (u >= th[k0 + 1] ? 1u : 0u);
  return up ? (N - 1u) - c : c;
}

// Code of a level-1 angle of the pair (x, y) = (y_{2i}, y_{2i+1}); t1a, t1b = tan^2
// of the first and third edges inside a quadrant (4-bit grids; the middle edge,
// pi/4, is the exact test sv >= su).  Branch-free.
template <int BITS>
__device__ __forceinline__ uint32_t code_level1(float x, float y, float t1a, float t1b) {
  constexpr uint32_t M = (1u << BITS) / 4;  // cells per quadrant
  // quadrant of (u, v) = (-x, -y): 0: u > 0, v >= 0; 1: u <= 0, v > 0; 2: u < 0, v <= 0;
  // 3: u >= 0, v < 0; a pair of two zeros has theta = 0, i.e. phi = pi: code 2M
  const uint32_t q1 = (x >= 0.0f && y < 0.0f) ? 1u : 0u;
  const uint32_t q2 = (x > 0.0f && y >= 0.0f) ? 2u : 0u;
  const uint32_t q3 = (x <= 0.0f && y > 0.0f) ? 3u : 0u;
  const uint32_t quad = q1 | q2 | q3;
  // rotated into the first quadrant: (u', v') = (u, v), (v, -u), (-u, -v), (-v, u)
  const float xx = x * x, yy = y * y;
  const bool swap = quad & 1u;
  const float su = swap ? yy : xx, sv = swap ? xx : yy;
  uint32_t sub = 0;
  if constexpr (M == 2) sub = sv >= su ? 1u : 0u;
  if constexpr (M == 4) {
    sub = sv >= su ? 2u : 0u;
    sub += sv >= su * (sub ? t1b : t1a) ? 1u : 0u;
  }
  const uint32_t code = quad * M + sub;
  return (x == 0.0f && y == 0.0f) ? 2 * M : code;
}

__device__ __forceinline__ uint16_t f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// ------------------------------------------------------------------ append

struct PolarAppendArgs {
  const void* x;          // [n_tok][H][d] fp32 or bf16
  const int64_t* slots;   // [n_tok]
  int64_t n_vec;          // n_tok * H
  int H;
  int64_t max_slot;
  uint8_t* pool;
  int page_bytes;
  const float* signs;     // [d] +-1
  unsigned* status;
  PolarGrid grid;
};

// The 32 record slots [32q, 32q + 32) of one vector, one code per byte (4 words),
// packed to the BITS-bit bitstream: BITS words.
template <int BITS>
__device__ __forceinline__ void pack_slots(const uint32_t (&b)[8], uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {  // bytes b0..b3 -> nibble pairs, two input words per output word
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t t0 = b[2 * k] | (b[2 * k] >> 4), t1 = b[2 * k + 1] | (b[2 * k + 1] >> 4);
      w[k] = __byte_perm(t0, t1, 0x6420u);
    }
  } else {
    uint32_t code[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) code[i] = (b[i >> 2] >> (8 * (i & 3))) & 0xFFu;
    pack32<BITS>(code, w);
  }
}

// Lane q of a quad holds the 32 rotated coordinates [32q, 32q + 32) of one vector.
// The codes go through a per-vector byte array in shared memory (slot order), from
// which lane q packs and stores record bits [32 BITS q, 32 BITS (q + 1)).
template <int BITS, typename TIn>
__global__ void __launch_bounds__(256, 3) k_polar_append(PolarAppendArgs a) {
  __shared__ float s_th[16];
  __shared__ uint8_t s_ucell[256];
  __shared__ __align__(16) uint8_t s_codes[8][8][128];  // [warp][vector of the warp][slot]
  if (threadIdx.x < 16) s_th[threadIdx.x] = a.grid.th[threadIdx.x];
  s_ucell[threadIdx.x] = a.grid.ucell[threadIdx.x];  // 256 threads
  __syncthreads();
  const int lane = threadIdx.x & 31, q = lane & 3;
  uint8_t* rec_s = s_codes[threadIdx.x >> 5][lane >> 2];
  const float t1a = a.grid.t1[1], t1b = a.grid.t1[3];
  uint32_t sw = 0;  // sign flips of coordinates [32q, 32q + 32)
#pragma unroll
  for (int i = 0; i < 32; ++i) sw |= (__ldg(a.signs + 32 * q + i) < 0.0f ? 1u : 0u) << i;
  const int64_t nq = ((a.n_vec + 7) / 8) * 8;  // whole warps keep the quad shuffles convergent
  for (int64_t v0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2; v0 < nq;
       v0 += ((int64_t)gridDim.x * blockDim.x) >> 2) {
    const bool live = v0 < a.n_vec;
    const int64_t vec = live ? v0 : a.n_vec - 1;
    const int64_t tok = vec / a.H;
    const int head = (int)(vec - tok * a.H);
    const TIn* src = reinterpret_cast<const TIn*>(a.x) + vec * kD + 32 * q;
    float y[32];
    if constexpr (sizeof(TIn) == 2) {  // sign flips applied to the packed bf16 words
      const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(p + i);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 4 * i + k;  // word j: coordinates 2j, 2j + 1
          const uint32_t f = wv[k] ^ (((sw >> (2 * j)) & 1u) << 15 | ((sw >> (2 * j + 1)) & 1u) << 31);
          y[2 * j] = __uint_as_float(f << 16);
          y[2 * j + 1] = __uint_as_float(f & 0xFFFF0000u);
        }
      }
    } else {
      load32<TIn>(src, y);
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(__float_as_uint(y[i]) ^ (((sw >> i) & 1u) << 31));
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = fmaf(y[i], y[i], ss);
    const float norm = sqrtf(quad_sum(ss));
    fwht128_quad_f2(y, q);  // unnormalised: angles do not depend on the scale
    // level 1: 16 angles (4 code bytes per word), squared radii
    uint32_t b1[4] = {0u, 0u, 0u, 0u};
    float s[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      b1[i >> 2] |= code_level1<BITS>(y[2 * i], y[2 * i + 1], t1a, t1b) << (8 * (i & 3));
      s[i] = fmaf(y[2 * i], y[2 * i], y[2 * i + 1] * y[2 * i + 1]);
    }
    // levels 2..5 inside the lane: 8 + 4 + 2 + 1 angles
    uint32_t b2[2] = {0u, 0u}, b3 = 0u, b4 = 0u, c5;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      b2[i >> 2] |= code_high<BITS>(s[2 * i], s[2 * i + 1], s_th, s_ucell) << (8 * (i & 3));
      s[i] = s[2 * i] + s[2 * i + 1];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      b3 |= code_high<BITS>(s[2 * i], s[2 * i + 1], s_th, s_ucell) << (8 * i);
      s[i] = s[2 * i] + s[2 * i + 1];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      b4 |= code_high<BITS>(s[2 * i], s[2 * i + 1], s_th, s_ucell) << (8 * i);
      s[i] = s[2 * i] + s[2 * i + 1];
    }
    c5 = code_high<BITS>(s[0], s[1], s_th, s_ucell);
    const float s5 = s[0] + s[1];
    // levels 6 and 7 from the quad's four squared radii (every lane computes them)
    const int base = lane & ~3;
    const float r0 = __shfl_sync(0xffffffffu, s5, base), r1 = __shfl_sync(0xffffffffu, s5, base + 1);
    const float r2 = __shfl_sync(0xffffffffu, s5, base + 2), r3 = __shfl_sync(0xffffffffu, s5, base + 3);
    const uint32_t c6a = code_high<BITS>(r0, r1, s_th, s_ucell), c6b = code_high<BITS>(r2, r3, s_th, s_ucell);
    const uint32_t c7 = code_high<BITS>(r0 + r1, r2 + r3, s_th, s_ucell);
    // codes to the vector's byte array in slot order
    *reinterpret_cast<uint4*>(rec_s + 16 * q) = make_uint4(b1[0], b1[1], b1[2], b1[3]);  // level 1
    *reinterpret_cast<uint2*>(rec_s + 64 + 8 * q) = make_uint2(b2[0], b2[1]);            // level 2
    *reinterpret_cast<uint32_t*>(rec_s + 96 + 4 * q) = b3;                               // level 3
    *reinterpret_cast<uint16_t*>(rec_s + 112 + 2 * q) = (uint16_t)b4;                    // level 4
    rec_s[120 + q] = (uint8_t)c5;                                                        // level 5
    if (q == 0) *reinterpret_cast<uint32_t*>(rec_s + 124) = c6a | c6b << 8 | c7 << 16;  // 6, 7, pad
    __syncwarp();
    const uint4 lo = *reinterpret_cast<const uint4*>(rec_s + 32 * q);
    const uint4 hi = *reinterpret_cast<const uint4*>(rec_s + 32 * q + 16);
    __syncwarp();  // the array is rewritten by the next iteration
    const uint32_t bytes[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t w[BITS];
    pack_slots<BITS>(bytes, w);
    if (!live) continue;
    const int64_t slot = __ldg(a.slots + tok);
    if (slot < 0) continue;
    if (slot >= a.max_slot) {
      if (q == 0) flag_status(a.status, TQ_DEV_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot >> 4;
    const int off = (int)(slot & 15);
    uint8_t* page = a.pool + (blk * a.H + head) * (int64_t)a.page_bytes;
    uint8_t* rec = page + off * (16 * BITS) + q * (4 * BITS);
    if constexpr (BITS == 4) {
      *reinterpret_cast<uint4*>(rec) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (BITS == 3) {
      uint32_t* r32 = reinterpret_cast<uint32_t*>(rec);
      r32[0] = w[0];
      r32[1] = w[1];
      r32[2] = w[2];
    } else {
      *reinterpret_cast<uint2*>(rec) = make_uint2(w[0], w[1]);
    }
    if (q == 0) *reinterpret_cast<uint16_t*>(page + 16 * (16 * BITS) + 2 * off) = f16_bits(norm);
  }
}

// ------------------------------------------------------------------ decode / combine

// CTA per (sequence, query head), thread t = coordinate t.
template <typename TO>
__global__ void __launch_bounds__(128) k_polar_combine(const float* __restrict__ part, const float* __restrict__ ml,
                                                       int splits, const float* __restrict__ signs, TO* out) {
  __shared__ float red[4], y[kD];
  const int t = threadIdx.x;
  const int64_t bh = blockIdx.x;
  const float* mlr = ml + bh * splits * 2;
  float mx = -INFINITY;
  for (int s = t; s < splits; s += 128) mx = fmaxf(mx, mlr[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) red[t >> 5] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float acc = 0.0f, L = 0.0f;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ms = mlr[2 * s];
      if (ms == -INFINITY) continue;  // empty chunk
      const float f = exp2f(ms - M);
      acc = fmaf(part[(bh * splits + s) * kD + t], f, acc);
      L = fmaf(mlr[2 * s + 1], f, L);
    }
  }
  y[t] = L > 0.0f ? acc / L : 0.0f;
  __syncthreads();
  for (int h = 1; h < kD; h <<= 1) {  // y <- H y
    const bool lower = (t & h) == 0;
    float u = 0.0f, v = 0.0f;
    if (lower) { u = y[t]; v = y[t + h]; }
    __syncthreads();
    if (lower) { y[t] = u + v; y[t + h] = u - v; }
    __syncthreads();
  }
  store_elem<TO>(out + bh * kD + t, y[t] * kInvSqrtD * __ldg(signs + t));
}

// ------------------------------------------------------------------ dequantize

// Leaf writing a whole direction (times r) into a [32][128] tile row, quads at c ^ (v & 7).
struct RowLeaf {
  float4 buf;
  float* row;
  int sw;
  template <int J>
  __device__ __forceinline__ void at(float v) {
    constexpr int k = J & 3;
    if constexpr (k == 0) buf.x = v;
    if constexpr (k == 1) buf.y = v;
    if constexpr (k == 2) buf.z = v;
    if constexpr (k == 3) {
      buf.w = v;
      *reinterpret_cast<float4*>(row + (((J >> 2) ^ sw) << 2)) = buf;
    }
  }
};

// Two warps per CTA; a warp takes 32 vectors: lane v rebuilds r * y_hat of vector v into the tile,
// then the warp applies Pi^T = D H / sqrt(d) to each row (lane L: coordinates 4L..4L+3).
template <int BITS, typename TO>
__global__ void __launch_bounds__(64) k_polar_dequant(const uint8_t* __restrict__ pool, int H, int page_bytes,
                                                       int64_t max_slot, const int64_t* __restrict__ slots,
                                                       int64_t n_vec, const float* __restrict__ signs, TO* out,
                                                       unsigned* status, PolarGrid grid) {
  __shared__ float tabs[64];
  __shared__ __align__(16) float tiles[2][32 * 128];
  if (threadIdx.x < 32) {
    tabs[threadIdx.x] = grid.cs1[threadIdx.x];
    tabs[32 + threadIdx.x] = grid.csh[threadIdx.x];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* tile = tiles[warp];
  float sg[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) sg[k] = __ldg(signs + 4 * lane + k) * kInvSqrtD;
  const int64_t n_groups = (n_vec + 31) / 32;
  for (int64_t grp = (int64_t)blockIdx.x * 2 + warp; grp < n_groups; grp += (int64_t)gridDim.x * 2) {
    const int64_t vec = grp * 32 + lane;
    float r = 0.0f;
    uint32_t w[16] = {};
    if (vec < n_vec) {
      const int64_t tok = vec / H;
      const int head = (int)(vec - tok * H);
      const int64_t slot = __ldg(slots + tok);
      if (slot >= max_slot) flag_status(status, TQ_DEV_BAD_SLOT);
      if (slot >= 0 && slot < max_slot) {
        const uint8_t* page = pool + ((slot >> 4) * H + head) * (int64_t)page_bytes;
        const int off = (int)(slot & 15);
        const uint4* rec = reinterpret_cast<const uint4*>(page + off * (16 * BITS));
#pragma unroll
        for (int c = 0; c < BITS; ++c) {
          const uint4 v = __ldg(rec + c);
          w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
        r = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(page + 16 * (16 * BITS) + 2 * off)));
      }
    }
    RowLeaf rl;
    rl.row = tile + lane * 128;
    rl.sw = lane & 7;
    expand<BITS, 7, 0>(w, r, tabs, tabs + 32, rl);
    __syncwarp();
    const int64_t rem = n_vec - grp * 32;
    const int nv = rem < 32 ? (int)rem : 32;
    for (int v = 0; v < nv; ++v) {
      const float4 t4 = *reinterpret_cast<const float4*>(tile + v * 128 + ((lane ^ (v & 7)) << 2));
      float y[4] = {t4.x, t4.y, t4.z, t4.w};
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
      TO* dst = out + (grp * 32 + v) * kD + 4 * lane;
#pragma unroll
      for (int k = 0; k < 4; ++k) store_elem<TO>(dst + k, y[k] * sg[k]);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ launchers

template <int BITS>
static cudaError_t run_polar_append(const PolarAppendArgs& a, bool f32, int num_sms, cudaStream_t st) {
  const int64_t threads = ((a.n_vec + 7) / 8) * 32;
  int64_t grid = (threads + 255) / 256;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  if (grid < 1) grid = 1;
  if (f32) k_polar_append<BITS, float><<<(unsigned)grid, 256, 0, st>>>(a);
  else k_polar_append<BITS, __nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_polar_append(const tq_cache_desc& d, int which, const void* x, int in_dtype,
                                const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  const int bits = which == 0 ? d.fmt.bits_k : d.fmt.bits_v;
  PolarAppendArgs a;
  a.x = x;
  a.slots = slots;
  a.n_vec = n_tok * d.num_kv_heads;
  a.H = d.num_kv_heads;
  a.max_slot = d.num_blocks * kBlock;
  a.pool = reinterpret_cast<uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  a.page_bytes = (int)page_bytes_of(d, which);
  a.signs = d.rotation;
  a.status = status;
  a.grid = polar_grid(bits);
  const bool f32 = in_dtype == TQ_F32;
  switch (bits) {
    case 2: return run_polar_append<2>(a, f32, num_sms, st);
    case 3: return run_polar_append<3>(a, f32, num_sms, st);
    default: return run_polar_append<4>(a, f32, num_sms, st);
  }
}

template <int BITS, typename TO>
static cudaError_t run_polar_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n_vec,
                                     TO* out, unsigned* status, int num_sms, cudaStream_t st) {
  const int64_t groups = (n_vec + 31) / 32;
  int64_t grid = (groups + 1) / 2;
  if (grid > (int64_t)num_sms * 6) grid = (int64_t)num_sms * 6;
  if (grid < 1) grid = 1;
  k_polar_dequant<BITS, TO><<<(unsigned)grid, 64, 0, st>>>(
      reinterpret_cast<const uint8_t*>(which == 0 ? d.k_cache : d.v_cache), d.num_kv_heads,
      (int)page_bytes_of(d, which), d.num_blocks * kBlock, slots, n_vec, d.rotation, out, status,
      polar_grid(which == 0 ? d.fmt.bits_k : d.fmt.bits_v));
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_polar_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n, void* out,
                                 int out_dtype, unsigned* status, int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t n_vec = n * d.num_kv_heads;
  const int bits = which == 0 ? d.fmt.bits_k : d.fmt.bits_v;
  if (out_dtype == TQ_F32) {
    float* o = reinterpret_cast<float*>(out);
    switch (bits) {
      case 2: return run_polar_dequant<2>(d, which, slots, n_vec, o, status, num_sms, st);
      case 3: return run_polar_dequant<3>(d, which, slots, n_vec, o, status, num_sms, st);
      default: return run_polar_dequant<4>(d, which, slots, n_vec, o, status, num_sms, st);
    }
  }
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
  switch (bits) {
    case 2: return run_polar_dequant<2>(d, which, slots, n_vec, o, status, num_sms, st);
    case 3: return run_polar_dequant<3>(d, which, slots, n_vec, o, status, num_sms, st);
    default: return run_polar_dequant<4>(d, which, slots, n_vec, o, status, num_sms, st);
  }
}

cudaError_t launch_polar_decode(const DecodeCall& c, cudaStream_t st) {
  const tq_cache_desc& d = *c.desc;
  const DecodeWorkspace ws = decode_workspace(c.batch, c.num_q_heads, c.splits, kD, false);
  PolarDecodeArgs a;
  a.kpool = reinterpret_cast<const uint8_t*>(d.k_cache);
  a.vpool = reinterpret_cast<const uint8_t*>(d.v_cache);
  a.kpage = (int)page_bytes_of(d, 0);
  a.vpage = (int)page_bytes_of(d, 1);
  a.Hkv = d.num_kv_heads;
  a.Hq = c.num_q_heads;
  a.g = c.num_q_heads / d.num_kv_heads;
  const int nh = a.g <= 4 ? 4 : 8;
  a.ngroups = (a.g + nh - 1) / nh;
  a.splits = c.splits;
  a.num_blocks = d.num_blocks;
  a.block_table = c.block_table;
  a.max_blocks = c.max_blocks;
  a.ctx_lens = c.ctx_lens;
  a.q = c.q;
  a.q_bf16 = c.q_dtype == TQ_BF16 ? 1 : 0;
  a.q_scale = c.sm_scale * kPolarLog2e * kInvSqrtD;
  a.signs = d.rotation;
  a.part = reinterpret_cast<float*>(c.workspace + ws.part_off);
  a.ml = reinterpret_cast<float*>(c.workspace + ws.ml_off);
  a.chunks = (int64_t)c.batch * d.num_kv_heads * a.ngroups * c.splits;
  a.status = c.status;
  const PolarGrid gk = polar_grid(d.fmt.bits_k), gv = polar_grid(d.fmt.bits_v);
  for (int i = 0; i < 32; ++i) {
    a.cs1k[i] = gk.cs1[i];
    a.cshk[i] = gk.csh[i];
    a.cs1v[i] = gv.cs1[i];
    a.cshv[i] = gv.csh[i];
  }
  cudaError_t e;
  switch (d.fmt.bits_k) {
    case 2: e = polar_decode_bk<2>(a, d.fmt.bits_v, nh, st); break;
    case 3: e = polar_decode_bk<3>(a, d.fmt.bits_v, nh, st); break;
    default: e = polar_decode_bk<4>(a, d.fmt.bits_v, nh, st); break;
  }
  if (e != cudaSuccess) return e;
  const unsigned cgrid = (unsigned)((int64_t)c.batch * c.num_q_heads);
  if (c.out_dtype == TQ_F32)
    k_polar_combine<float><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, d.rotation, reinterpret_cast<float*>(c.out));
  else
    k_polar_combine<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a.part, a.ml, c.splits, d.rotation,
                                                          reinterpret_cast<__nv_bfloat16*>(c.out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace tq
