// Quantize-on-append, the quantizer on given rotated coordinates, bf16-layer
// append and dequantization (libtq, sm_103a).
//
// Method (issoh.co.jp TurboQuant overview, §第1段 and §第2段; lilting.ch
// TurboQuant article, QJL section): per vector x, n = ||x||, y = Pi x / n,
// idx_j = #{i : y_j >= beta_i}, gamma = n / ||c[idx]|| (norm correction),
// LSB-first bit packing into the paged record, optional 1-bit QJL residual
// sigma = [S (Pi x - gamma c[idx]) >= 0] with rho = ||Pi x - gamma c[idx]||.
//
// Thread layout: 4 consecutive lanes (a quad) own one vector, lane q of the
// quad holding coordinates [32q, 32q + 32) in registers.  The Hadamard
// rotation is a fast Walsh-Hadamard transform: 5 butterfly stages inside the
// registers and 2 through quad shuffles.  A CTA of 256 threads handles tiles
// of 64 vectors in a grid-stride loop.  Dense rotations and the QJL projection
// are 128x128 mat-vecs against a padded copy of the matrix in shared memory.
#include <cuda_fp8.h>

#include <cmath>
#include <cstring>

#include "tq_async.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tcgen05.cuh"

namespace tq {

enum { MODE_HADAMARD = 0, MODE_DENSE = 1, MODE_GIVEN_Y = 2 };

struct QuantArgs {
  const void* x;         // [n_tok][H][d] input vectors (MODE_HADAMARD / MODE_DENSE)
  const float* y;        // [n_tok][H][d] rotated unit coordinates (MODE_GIVEN_Y)
  const float* norms;    // [n_tok][H] norms (MODE_GIVEN_Y)
  const int64_t* slots;  // [n_tok]
  int64_t n_vec;         // n_tok * H
  int H;
  int64_t max_slot;      // num_blocks * 16
  uint8_t* pool;
  int page_bytes;
  const float* rot;      // signs[d] or Pi[d][d]
  const float* qjl;      // S[d][d]
  Codebook cb;
  int norm_mode;
  unsigned* status;
  // Keys and values of one append share a launch when their formats and tables
  // agree: blocks with blockIdx.y = 1 read x_v and write pool_v instead.
  const void* x_v;
  uint8_t* pool_v;
};

constexpr int kTile = 64;            // vectors per CTA iteration
constexpr int kThreads = 256;
constexpr int kTileStride = kD + 4;  // padded row of the vector tile (floats)
constexpr int kPadQ = 36;            // padded quarter-row of a staged matrix (floats)
constexpr size_t kTableBytes = 4096;
constexpr size_t kTileBytes = (size_t)kTile * kTileStride * 4;
constexpr size_t kMatBytes = (size_t)kD * 4 * kPadQ * 4;

// Cell table of the quantizer for rotated coordinates (|y| <= 1 up to rounding).
// t = fmaf(y, 63, 1.5 * 2^16 + 64) has an ulp of 2^-7, so bits 7..13 of t are
// cell(y) = floor(63 y + 64 + <2^-7 rounding>): a monotone map of [-1, 1] onto
// cells 1..127, each narrower (1/63) than the smallest gap between boundaries of
// the supported codebooks, so a cell holds at most one boundary P.  For y in cell
// i, idx = #{beta <= y} = base_i + [y >= P_i] exactly (the boundaries' own cells
// come from the same fmaf).  Entry = {P, c[base]^2, c[base + 1]^2, base}; 8
// interleaved copies (one per lane of a quarter warp) make a 128-byte row per
// cell, so bits 7..13 of t are the row offset: with the table 16 KB aligned, one
// bitwise op turns t into the lane's entry address, and lookups never conflict.
constexpr int kQCells = 128;
constexpr float kQScale = 63.0f;
constexpr float kQMagic = 98304.0f + 64.0f;  // 1.5 * 2^16 + 64
constexpr size_t kLutQBytes = (size_t)kQCells * 8 * 16;
constexpr uint32_t kQRowMask = (uint32_t)(kQCells - 1) << 7;

__host__ __device__ __forceinline__ uint32_t qcell_bits(float y) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(fmaf(y, kQScale, kQMagic));
#else
  const float t = std::fmaf(y, kQScale, kQMagic);
  uint32_t u;
  std::memcpy(&u, &t, 4);
  return u;
#endif
}
__host__ __device__ __forceinline__ uint32_t qcell(float y) { return (qcell_bits(y) & kQRowMask) >> 7; }

// Host: every boundary of the table falls in its own cell, none in the end cells.
bool cell_table_ok(const float* boundaries, int nb) {
  for (int k = 0; k < nb; ++k) {
    const uint32_t ck = qcell(boundaries[k]);
    if (ck == 0u || ck == (uint32_t)(kQCells - 1)) return false;
    if (k > 0 && ck == qcell(boundaries[k - 1])) return false;
  }
  return true;
}

// dst[r][q][k] = transpose ? src[32q + k][r] : src[r][32q + k]   (src row-major d x d)
// (a CTA of kThreads threads; each thread's loads go out in batches, in flight together
// before their stores)
__device__ void stage_matrix(const float* __restrict__ src, float* dst, bool transpose) {
  if (transpose && (reinterpret_cast<uintptr_t>(src) & 15u) == 0u) {
    // lane = source row (mod 32), so the transposed stores of a warp hit 32 banks
    constexpr int kWarps = kThreads / 32, kCols = kD / 4 / kWarps;  // float4 columns per warp
    static_assert(kCols * kWarps * 4 == kD, "whole float4 columns");
    const int lane = threadIdx.x & 31, wq = threadIdx.x >> 5;
#pragma unroll
    for (int rb = 0; rb < kD / 32; ++rb) {  // source rows 32 rb + lane
      float4 v[kCols];
#pragma unroll
      for (int cb = 0; cb < kCols; ++cb)
        v[cb] = __ldg(reinterpret_cast<const float4*>(src) + (lane + 32 * rb) * (kD / 4) + wq + kWarps * cb);
#pragma unroll
      for (int cb = 0; cb < kCols; ++cb) {  // src[i][4 jq + t] -> dst row r = 4 jq + t, column c = i
        const int jq = wq + kWarps * cb;
        float* d0 = dst + (16 * jq + rb) * kPadQ + lane;
        d0[0] = v[cb].x;
        d0[4 * kPadQ] = v[cb].y;
        d0[8 * kPadQ] = v[cb].z;
        d0[12 * kPadQ] = v[cb].w;
      }
    }
  } else {
    constexpr int kS = kD * kD / kThreads;  // floats per thread; consecutive threads, consecutive j
    static_assert(kS % 16 == 0 && kS * kThreads == kD * kD, "whole batches");
#pragma unroll
    for (int b0 = 0; b0 < kS; b0 += 16) {
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = __ldg(src + threadIdx.x + (b0 + k) * kThreads);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int e = (int)threadIdx.x + (b0 + k) * kThreads;
        const int i = e / kD, j = e % kD;  // src[i][j]
        const int r = transpose ? j : i;
        const int c = transpose ? i : j;
        dst[(r * 4 + (c >> 5)) * kPadQ + (c & 31)] = v[k];
      }
    }
  }
}

// out[k] = sum_r Mp[r][q][k] * vin[r]  for the 32 outputs of quarter q.
__device__ __forceinline__ void matvec_padded(const float* Mp, const float* vin, int q, float (&out)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) out[k] = 0.0f;
#pragma unroll 2
  for (int r = 0; r < kD; ++r) {
    const float v = vin[r];
    const float4* row = reinterpret_cast<const float4*>(Mp + (r * 4 + q) * kPadQ);
#pragma unroll
    for (int k4 = 0; k4 < 8; ++k4) {
      const float4 m = row[k4];
      out[4 * k4] = fmaf(m.x, v, out[4 * k4]);
      out[4 * k4 + 1] = fmaf(m.y, v, out[4 * k4 + 1]);
      out[4 * k4 + 2] = fmaf(m.z, v, out[4 * k4 + 2]);
      out[4 * k4 + 3] = fmaf(m.w, v, out[4 * k4 + 3]);
    }
  }
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float flip_sign(float v, uint32_t word, int bit) {
  return __uint_as_float(__float_as_uint(v) ^ ((word << (31 - bit)) & 0x80000000u));
}

// Three CTAs per SM for the plain Hadamard path: the append is latency bound, so
// residency matters more than the few registers the bound takes away.
template <int BITS, typename TIn, int MODE, bool QJL>
__global__ void __launch_bounds__(kThreads, (MODE == MODE_HADAMARD && !QJL) ? 3 : 1) k_quantize(QuantArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent decode may start its prologue
  const void* const x_in = blockIdx.y ? a.x_v : a.x;
  uint8_t* const pool = blockIdx.y ? a.pool_v : a.pool;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int H = 1 << (BITS - 1);
  constexpr int R = 16 * BITS;  // record bytes
  float* mag2 = reinterpret_cast<float*>(smem_raw);              // [H][32]
  float* ctab = mag2 + 8 * 32;                                   // [2H][32]
  uint32_t* signw = reinterpret_cast<uint32_t*>(ctab + 16 * 32);  // [4]
  constexpr bool LUTQ = MODE != MODE_GIVEN_Y;  // |y| <= 1 only for coordinates this kernel rotates
  // the cell table starts at the first 16 KB aligned shared address past the small tables
  const uint32_t smem_base = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t qtab_addr = (smem_base + (uint32_t)kTableBytes + 16383u) & ~16383u;
  float4* qtab = reinterpret_cast<float4*>(smem_raw + (qtab_addr - smem_base));  // [kQCells][8]
  unsigned char* const dyn = LUTQ ? smem_raw + (qtab_addr - smem_base) + kLutQBytes : smem_raw + kTableBytes;
  float* tile = reinterpret_cast<float*>(dyn);
  float* matP = reinterpret_cast<float*>(dyn + kTileBytes);
  float* matS = reinterpret_cast<float*>(dyn + kTileBytes + (MODE == MODE_DENSE ? kMatBytes : 0));

  const int tid = threadIdx.x, lane = tid & 31, q = tid & 3, vl = tid >> 2;
  for (int i = tid; i < H * 32; i += kThreads) {
    const float c = a.cb.c[H + i / 32];
    mag2[i] = c * c;
  }
  if (QJL)
    for (int i = tid; i < 2 * H * 32; i += kThreads) ctab[i] = a.cb.c[i / 32];
  if (MODE == MODE_HADAMARD && tid < 32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t m = __ballot_sync(0xffffffffu, __ldg(a.rot + 32 * k + lane) < 0.0f);
      if (lane == 0) signw[k] = m;
    }
  }
  if (MODE == MODE_DENSE) stage_matrix(a.rot, matP, /*transpose=*/true);  // out = Pi x
  if (QJL) stage_matrix(a.qjl, matS, /*transpose=*/true);                 // out = S r
  if (LUTQ) {  // the host checked that no cell holds two boundaries (cell_table_ok)
    if (tid < kQCells) {
      constexpr int NB = (1 << BITS) - 1;  // boundaries
      uint32_t base = 0u;
      float P = INFINITY;
      for (int k = 0; k < NB; ++k) {
        const float bk = a.cb.b[k];
        const uint32_t ck = qcell(bk);
        if (ck < (uint32_t)tid) ++base;
        if (ck == (uint32_t)tid) P = bk;
      }
      const float c0 = a.cb.c[min(base, (uint32_t)NB)];
      const float c1 = a.cb.c[min(base + 1u, (uint32_t)NB)];
      const float4 e = make_float4(P, c0 * c0, c1 * c1, __uint_as_float(base));
#pragma unroll
      for (int r = 0; r < 8; ++r) qtab[tid * 8 + ((r + tid) & 7)] = e;  // rotated: no store conflicts
    }
  }
  __syncthreads();
  const uint32_t qrow_addr = qtab_addr | (16u * (uint32_t)(lane & 7));
  const uint32_t sw = (MODE == MODE_HADAMARD) ? signw[q] : 0u;
  // bf16 input, Hadamard: sign flips of coordinate pairs as masks on the packed bf16 words
  uint32_t pmask[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) pmask[j] = ((sw >> (2 * j)) & 1u) << 15 | ((sw >> (2 * j + 1)) & 1u) << 31;
  const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)

  const int64_t n_tiles = (a.n_vec + kTile - 1) / kTile;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t vec_raw = t * kTile + vl;
    const bool valid = vec_raw < a.n_vec;
    const int64_t vec = valid ? vec_raw : (a.n_vec - 1);

    float x[32];  // becomes Pi x (full scale) for the quad's 32 coordinates
    float n;
    if constexpr (MODE == MODE_GIVEN_Y) {
      load32<float>(a.y + vec * kD + 32 * q, x);
      n = __ldg(a.norms + vec);
    } else {
      constexpr bool kBf16Signs = MODE == MODE_HADAMARD && sizeof(TIn) == 2;
      if constexpr (kBf16Signs) {  // widen with the sign flips applied to the packed words
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const TIn*>(x_in) + vec * kD + 32 * q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = __ldg(src + k);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t f = w[e] ^ pmask[4 * k + e];
            x[8 * k + 2 * e] = __uint_as_float(f << 16);
            x[8 * k + 2 * e + 1] = __uint_as_float(f & 0xFFFF0000u);
          }
        }
      } else {
        load32<TIn>(reinterpret_cast<const TIn*>(x_in) + vec * kD + 32 * q, x);
      }
      float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 xi = make_float2(x[2 * i], x[2 * i + 1]);
        ss2 = __ffma2_rn(xi, xi, ss2);
      }
      n = sqrtf(quad_sum(ss2.x + ss2.y));
      if constexpr (MODE == MODE_HADAMARD) {
        if constexpr (!kBf16Signs) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = flip_sign(x[i], sw, i);
        }
        fwht128_quad_f2(x, q);  // unnormalised: H D x = sqrt(d) Pi x
        if constexpr (QJL) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] *= inv_sqrt_d;
        }
      } else {
        __syncthreads();  // previous iteration is done with the tile
#pragma unroll
        for (int i = 0; i < 32; ++i) tile[vl * kTileStride + 32 * q + i] = x[i];
        __syncthreads();
        matvec_padded(matP, tile + vl * kTileStride, q, x);
      }
    }
    // y = (Pi x) / n; MODE_GIVEN_Y already holds y and uses it as is.  Without QJL the
    // Hadamard path keeps H D x unnormalised and folds 1 / sqrt(d) in here.
    constexpr bool kUnnorm = MODE == MODE_HADAMARD && !QJL;
    const float inv_n = (MODE == MODE_GIVEN_Y) ? 1.0f : (n > 0.0f ? (kUnnorm ? inv_sqrt_d : 1.0f) / n : 0.0f);

    uint32_t code[32];
    float c2 = 0.0f;
    if constexpr (LUTQ) {
      float2 c2v = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 y = __fmul2_rn(make_float2(x[i], x[i + 1]), make_float2(inv_n, inv_n));
        const float4 e0 = lds128f((qcell_bits(y.x) & kQRowMask) | qrow_addr);
        const float4 e1 = lds128f((qcell_bits(y.y) & kQRowMask) | qrow_addr);
        const bool up0 = y.x >= e0.x, up1 = y.y >= e1.x;
        code[i] = __float_as_uint(e0.w) + (up0 ? 1u : 0u);
        code[i + 1] = __float_as_uint(e1.w) + (up1 ? 1u : 0u);
        c2v = __fadd2_rn(c2v, make_float2(up0 ? e0.z : e0.y, up1 ? e1.z : e1.y));
      }
      c2 = c2v.x + c2v.y;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float y = (MODE == MODE_GIVEN_Y) ? x[i] : x[i] * inv_n;
        int mag;
        code[i] = quantize_coord<BITS>(y, a.cb, &mag);
        c2 += mag2[mag * 32 + lane];
      }
    }
    c2 = quad_sum(c2);
    float gamma;
    if (a.norm_mode == TQ_NORM_RAW) gamma = n;
    else gamma = (n > 0.0f && c2 > 0.0f) ? n / sqrtf(c2) : 0.0f;

    uint32_t sbits = 0u;
    float rho = 0.0f;
    if constexpr (QJL) {
      float rr = 0.0f;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float r = x[i] - gamma * ctab[code[i] * 32 + lane];
        rr = fmaf(r, r, rr);
        tile[vl * kTileStride + 32 * q + i] = r;
      }
      rho = sqrtf(quad_sum(rr));
      __syncthreads();
      float z[32];
      matvec_padded(matS, tile + vl * kTileStride, q, z);
#pragma unroll
      for (int i = 0; i < 32; ++i) sbits |= (z[i] >= 0.0f ? 1u : 0u) << i;
    }

    const int64_t tok = vec / a.H;
    const int head = (int)(vec - tok * a.H);
    const int64_t slot = __ldg(a.slots + tok);
    if (valid && slot >= a.max_slot) {
      if (q == 0) flag_status(a.status, TQ_DEV_BAD_SLOT);
    } else if (valid && slot >= 0) {
      const int64_t blk = slot >> 4;
      const int off = (int)(slot & 15);
      uint8_t* page = pool + (blk * a.H + head) * (int64_t)a.page_bytes;
      uint32_t w[BITS];
      pack32<BITS>(code, w);
      uint8_t* rec = page + off * R;
      if constexpr (BITS == 4) {
        *reinterpret_cast<uint4*>(rec + 16 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      } else if constexpr (BITS == 2) {
        *reinterpret_cast<uint2*>(rec + 8 * q) = make_uint2(w[0], w[1]);
      } else {
        uint32_t* r32 = reinterpret_cast<uint32_t*>(rec + 12 * q);
        r32[0] = w[0]; r32[1] = w[1]; r32[2] = w[2];
      }
      if (q == 0) *reinterpret_cast<float*>(page + 16 * R + 4 * off) = gamma;
      if constexpr (QJL) {
        *reinterpret_cast<uint32_t*>(page + 16 * R + 64 + 16 * off + 4 * q) = sbits;
        if (q == 0) *reinterpret_cast<float*>(page + 16 * R + 64 + 256 + 4 * off) = rho;
      }
    }
  }
}

// ------------------------------------------------- bf16 Hadamard append, staged
//
// The same quantizer for bf16 inputs on the Hadamard path without QJL, laid out
// so that one lane owns one whole vector: all seven butterfly stages of the FWHT
// run in registers (no shuffles), on float pairs v[j] = (x_j, x_{j+64}) so that
// six of them are packed fp32-pair operations.  Each warp streams tiles of 32
// vectors through its own shared-memory stage with 2-D tensor copies
// (two boxes of [32 vectors][64 coordinates], 128-byte swizzle: lane l reads
// 16-byte chunk c of its row at chunk c ^ (l & 7), so no read conflicts).  The
// stage is refilled with the warp's next tile as soon as the current one is in
// registers, so that tile's copy overlaps the current tile's arithmetic.
// The cell entries shrink to 8 bytes {P, base} (one 64-bit read per
// coordinate); the norm-correction sum sum_j c[idx_j]^2 is read per pair of
// codes from a table of c[lo]^2 + c[hi]^2 indexed by the packed pair.
constexpr int kTW = 12;                       // warps per CTA (3 per scheduler: 168 registers)
constexpr int kTStages = 1;                   // tiles per warp ring: refilled as soon as unpacked
constexpr uint32_t kTBox = 32 * 128;          // one box: 32 vectors x 64 bf16 coordinates
constexpr uint32_t kTStage = 2 * kTBox;       // 32 whole vectors
constexpr uint32_t kTCellBytes = 128 * 128;   // [cell][16 replicas] {P, base}
constexpr uint32_t kTPairBytes = 256 * 128;   // [pair][32 replicas] c[lo]^2 + c[hi]^2
constexpr uint32_t kTMiscBytes = 1024;        // sign masks (256 B) and mbarriers
constexpr size_t kTSmem = 16384 + kTCellBytes + kTPairBytes + kTMiscBytes + (size_t)kTW * kTStages * kTStage;

struct QuantTmaArgs {
  CUtensorMap tm[2];  // [n_vec][128] bf16 keys / values: box [32][64], 128-byte swizzle
  uint8_t* pool[2];
  const int64_t* slots;
  int64_t tiles;      // 32-vector tiles per tensor
  uint32_t n_vec;     // vectors per tensor (n_tok * H)
  int ny;             // tensors in this launch (1, or 2 for keys and values)
  int H;
  int page_bytes;
  int64_t max_slot;
  const float* rot;   // signs[128]
  Codebook cb;
  int norm_mode;
  unsigned* status;
};

__device__ __forceinline__ uint4 lds128u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t addr) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Tables of the one-lane-per-vector kernels (threads 0 .. max(128, NC^2) - 1 write):
//   cell table, 128 rows of 16 replicas of {P, base} (8 B; the host checked that no
//   cell holds two boundaries), at a 16 KB aligned shared address;
//   pair table, NC^2 rows of 32 replicas of c[lo]^2 + c[hi]^2 for pair lo + NC * hi.
template <int BITS>
__device__ __forceinline__ void build_pair_cell_tables(const Codebook& cb, unsigned char* cell, unsigned char* pair) {
  constexpr int NC = 1 << BITS, NB = NC - 1;
  const int tid = threadIdx.x;
  if (tid < 128) {
    uint32_t base = 0u;
    float P = INFINITY;
    for (int k = 0; k < NB; ++k) {
      const float bk = cb.b[k];
      const uint32_t ck = qcell(bk);
      if (ck < (uint32_t)tid) ++base;
      if (ck == (uint32_t)tid) P = bk;
    }
    float2* row = reinterpret_cast<float2*>(cell + tid * 128);
#pragma unroll
    for (int r = 0; r < 16; ++r) row[(r + tid) & 15] = make_float2(P, __uint_as_float(base));  // rotated: no conflicts
  }
  if (tid < NC * NC) {
    const float lo = cb.c[tid & (NC - 1)], hi = cb.c[tid / NC];
    const float v = lo * lo + hi * hi;
    float4* row = reinterpret_cast<float4*>(pair + tid * 128);
#pragma unroll
    for (int r = 0; r < 8; ++r) row[(r + tid) & 7] = make_float4(v, v, v, v);
  }
}

// Codes of the coordinate pair held in x (already H D x, unnormalised), scaled by s.
__device__ __forceinline__ void quant_pair(float2 x, float2 s, uint32_t qrow, uint32_t& c0, uint32_t& c1) {
  const float2 y = __fmul2_rn(x, s);
  const float2 t = __ffma2_rn(y, make_float2(kQScale, kQScale), make_float2(kQMagic, kQMagic));
  const float2 e0 = lds64f((__float_as_uint(t.x) & kQRowMask) | qrow);
  const float2 e1 = lds64f((__float_as_uint(t.y) & kQRowMask) | qrow);
  c0 = __float_as_uint(e0.y) + (y.x >= e0.x ? 1u : 0u);
  c1 = __float_as_uint(e1.y) + (y.y >= e1.x ? 1u : 0u);
}

// The record of one vector held as coordinate pairs v[j] = (x_j, x_{j+64}) (the
// staged kernel's layout after its FWHT), scaled by s2: the LSB-first record
// words of the codes, and ||c[idx]||^2 summed through the pair table (returned).
template <int BITS>
__device__ __forceinline__ float cell_record_split(const float2 (&v)[64], float2 s2, uint32_t qrow, uint32_t prow,
                                                   uint32_t (&wd)[4 * BITS]) {
  float2 c2p[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
  if constexpr (BITS == 4) {
#pragma unroll
    for (int j = 0; j < 64; j += 8) {
      uint32_t bx[4], by[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t x0, y0, x1, y1;
        quant_pair(v[j + 2 * k], s2, qrow, x0, y0);
        quant_pair(v[j + 2 * k + 1], s2, qrow, x1, y1);
        bx[k] = x0 | (x1 << 4);  // codes of coordinates j + 2k, j + 2k + 1
        by[k] = y0 | (y1 << 4);  // ... and of the same plus 64
        c2p[k & 1] = __fadd2_rn(c2p[k & 1], make_float2(lds32f(prow + (bx[k] << 7)), lds32f(prow + (by[k] << 7))));
      }
      wd[j / 8] = __byte_perm(__byte_perm(bx[0], bx[1], 0x0040), __byte_perm(bx[2], bx[3], 0x0040), 0x5410);
      wd[8 + j / 8] = __byte_perm(__byte_perm(by[0], by[1], 0x0040), __byte_perm(by[2], by[3], 0x0040), 0x5410);
    }
  } else {
#pragma unroll
    for (int jb = 0; jb < 64; jb += 32) {
      uint32_t cx[32], cy[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) quant_pair(v[jb + i], s2, qrow, cx[i], cy[i]);
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        c2p[(i >> 1) & 1] = __fadd2_rn(c2p[(i >> 1) & 1], make_float2(lds32f(prow + ((cx[i] | (cx[i + 1] << BITS)) << 7)),
                                                                     lds32f(prow + ((cy[i] | (cy[i + 1] << BITS)) << 7))));
      uint32_t wx[BITS], wy[BITS];
      pack32<BITS>(cx, wx);
      pack32<BITS>(cy, wy);
#pragma unroll
      for (int k = 0; k < BITS; ++k) {
        wd[(jb / 32) * BITS + k] = wx[k];      // coordinates jb .. jb + 31
        wd[(2 + jb / 32) * BITS + k] = wy[k];  // coordinates 64 + jb .. 64 + jb + 31
      }
    }
  }
  return (c2p[0].x + c2p[1].x) + (c2p[0].y + c2p[1].y);
}

// Codes of the 32 consecutive coordinates y[0..32) of one vector (a chunk of the
// tensor-core kernel's accumulator columns), scaled by s2: their BITS record
// words, and their c[idx]^2 added to c2p through the pair table.
template <int BITS>
__device__ __forceinline__ void cell_chunk32(const float (&y)[32], float2 s2, uint32_t qrow, uint32_t prow,
                                             uint32_t (&wc)[BITS], float2& c2p) {
  uint32_t code[32];
#pragma unroll
  for (int j = 0; j < 32; j += 2) quant_pair(make_float2(y[j], y[j + 1]), s2, qrow, code[j], code[j + 1]);
#pragma unroll
  for (int j = 0; j < 32; j += 4)
    c2p = __fadd2_rn(c2p, make_float2(lds32f(prow + ((code[j] | (code[j + 1] << BITS)) << 7)),
                                      lds32f(prow + ((code[j + 2] | (code[j + 3] << BITS)) << 7))));
  pack32<BITS>(code, wc);
}

template <int BITS>
__global__ void __launch_bounds__(kTW * 32, 1) k_quantize_tma(const __grid_constant__ QuantTmaArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent decode may start its prologue
  constexpr int R = 16 * BITS;             // record bytes
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const uint32_t cell_addr = (sbase + 16383u) & ~16383u;  // 16 KB aligned: address = (t & mask) | row
  const uint32_t pair_addr = cell_addr + kTCellBytes;
  const uint32_t misc_addr = pair_addr + kTPairBytes;
  const uint32_t ring_addr = misc_addr + kTMiscBytes;     // 1 KB aligned (swizzled boxes)
  auto gen = [&](uint32_t addr) { return smem_raw + (addr - sbase); };

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gen(misc_addr + 256)) + w * kTStages;
  const int64_t total = a.tiles * a.ny;
  const int64_t gw = (int64_t)blockIdx.x * kTW + w, G = (int64_t)gridDim.x * kTW;
  const int64_t n_my = gw < total ? (total - gw + G - 1) / G : 0;
  const uint32_t ring = ring_addr + (uint32_t)w * kTStages * kTStage;

  // lane 0: 32 vectors of tile `it` of this warp into stage s (both boxes on one barrier)
  auto issue = [&](int64_t it, int s) {
    const int64_t tile = gw + it * G;
    const int kv = tile >= a.tiles ? 1 : 0;
    const int row = (int)((tile - kv * a.tiles) * 32);
    mbar_arrive_expect_tx(bar + s, kTStage);
    tensor_copy_2d(ring + (uint32_t)s * kTStage, &a.tm[kv], 0, row, bar + s);
    tensor_copy_2d(ring + (uint32_t)s * kTStage + kTBox, &a.tm[kv], 64, row, bar + s);
  };
  if (lane == 0) {
    for (int s = 0; s < kTStages; ++s) mbar_init(bar + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < kTStages && s < n_my; ++s) issue(s, s);
  }

  // tables, built while the first copies are in flight
  build_pair_cell_tables<BITS>(a.cb, gen(cell_addr), gen(pair_addr));
  if (tid < 64) {  // sign flips of coordinates 2k, 2k+1 as a mask on their packed bf16 word
    const uint32_t m = (__ldg(a.rot + 2 * tid) < 0.0f ? 0x8000u : 0u) | (__ldg(a.rot + 2 * tid + 1) < 0.0f ? 0x80000000u : 0u);
    *reinterpret_cast<uint32_t*>(gen(misc_addr + 4u * (uint32_t)tid)) = m;
  }
  __syncthreads();

  const uint32_t rowsw = ring + (uint32_t)lane * 128u + ((uint32_t)(lane & 7) << 4);  // row, swizzle bits
  const uint32_t qrow = cell_addr | ((uint32_t)(lane & 15) << 3);
  const uint32_t prow = pair_addr + ((uint32_t)lane << 2);
  const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
  const float2 m1 = make_float2(-1.0f, -1.0f);

  bool aborted = false;
  int64_t it = 0;
  for (; it < n_my; ++it) {
    const int s = (int)(it % kTStages);
    const uint32_t ph = (uint32_t)(it / kTStages) & 1u;
    const int64_t tile = gw + it * G;
    const int kv = tile >= a.tiles ? 1 : 0;
    const uint32_t vec = (uint32_t)((tile - kv * a.tiles) * 32) + (uint32_t)lane;
    const bool valid = vec < a.n_vec;
    const uint32_t tok = valid ? vec / (uint32_t)a.H : 0u;
    const int head = (int)(vec - tok * (uint32_t)a.H);
    const int64_t slot = valid ? __ldg(a.slots + tok) : -1;

    if (!mbar_wait(bar + s, ph)) {
      if (lane == 0) flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      aborted = true;
      break;
    }
    // widen with the sign flips applied: v[j] = (D x)_j, (D x)_{j+64}
    float2 v[64];
    const uint32_t sb = rowsw + (uint32_t)s * kTStage;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 d0 = lds128u(sb ^ ((uint32_t)c << 4));
      const uint4 d1 = lds128u((sb + kTBox) ^ ((uint32_t)c << 4));
      const uint4 p0 = lds128u(misc_addr + 16u * (uint32_t)c);
      const uint4 p1 = lds128u(misc_addr + 128u + 16u * (uint32_t)c);
      const uint32_t w0[4] = {d0.x ^ p0.x, d0.y ^ p0.y, d0.z ^ p0.z, d0.w ^ p0.w};
      const uint32_t w1[4] = {d1.x ^ p1.x, d1.y ^ p1.y, d1.z ^ p1.z, d1.w ^ p1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * c + 2 * e] = make_float2(__uint_as_float(w0[e] << 16), __uint_as_float(w1[e] << 16));
        v[8 * c + 2 * e + 1] = make_float2(__uint_as_float(w0[e] & 0xFFFF0000u), __uint_as_float(w1[e] & 0xFFFF0000u));
      }
    }
    __syncwarp();  // every lane has its tile in registers: the stage may be refilled
    if (lane == 0 && it + kTStages < n_my) {
      fence_proxy_async();
      issue(it + kTStages, s);
    }

    float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 64; ++j) ss2 = __ffma2_rn(v[j], v[j], ss2);
    const float n = sqrtf(ss2.x + ss2.y);

    // H D x, unnormalised: six stages over the bits of j, then the bit inside each pair
#pragma unroll
    for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        if ((j & h) == 0) {
          const float2 p = v[j], q = v[j + h];
          v[j] = __fadd2_rn(p, q);
          v[j + h] = __ffma2_rn(q, m1, p);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = make_float2(v[j].x + v[j].y, v[j].x - v[j].y);

    // y = Pi x / n = (H D x) / (sqrt(d) n)
    const float inv_n = n > 0.0f ? inv_sqrt_d / n : 0.0f;
    const float2 s2 = make_float2(inv_n, inv_n);
    uint32_t wd[4 * BITS];  // the record, LSB-first
    const float c2 = cell_record_split<BITS>(v, s2, qrow, prow, wd);
    float gamma;
    if (a.norm_mode == TQ_NORM_RAW) gamma = n;
    else gamma = (n > 0.0f && c2 > 0.0f) ? n / sqrtf(c2) : 0.0f;

    if (valid && slot >= a.max_slot) {
      flag_status(a.status, TQ_DEV_BAD_SLOT);
    } else if (valid && slot >= 0) {
      uint8_t* page = a.pool[kv] + ((slot >> 4) * a.H + head) * (int64_t)a.page_bytes;
      const int off = (int)(slot & 15);
      uint4* rec = reinterpret_cast<uint4*>(page + off * R);
#pragma unroll
      for (int k = 0; k < BITS; ++k) rec[k] = make_uint4(wd[4 * k], wd[4 * k + 1], wd[4 * k + 2], wd[4 * k + 3]);
      *reinterpret_cast<float*>(page + 16 * R + 4 * off) = gamma;
    }
  }
  if (aborted && lane == 0) {  // let copies still in flight into this warp's ring land before exiting
    for (int64_t k = it; k < n_my && k < it + kTStages; ++k) mbar_wait(bar + (int)(k % kTStages), (uint32_t)(k / kTStages) & 1u);
  }
  // Launched as a programmatic dependent (a batched append, or values after keys), this
  // grid touches no memory of the grid before it, but it must not complete before that
  // grid does: work queued after it relies on both.  (No-op for an ordinary launch.)
  grid_dep_wait();
}

// ------------------------------------- dense rotation append on tensor cores
//
// Batched appends of bf16 vectors through a dense Pi (Haar kind) are a GEMM:
// Y = X Pi^T for tiles of 128 vectors, M = N = K = 128.  Pi is split into bf16
// parts Pi = P_hi + P_lo + O(2^-16 |Pi|) (both K-major in shared memory, built
// once per CTA), and every K step of 16 issues two tcgen05.mma of kind::f16
// (X * P_hi^T, X * P_lo^T) into one fp32 accumulator of 128 tensor-memory
// columns.  Roles: warp 0 streams X tiles with 2-D tensor copies (boxes of
// [128 vectors][64 coordinates], 128-byte swizzle) into a 3-deep ring; one
// thread of warp 1 issues the MMAs; 16 epilogue warps in four groups serve four
// accumulators in turn (group e takes tiles e, e + 4, ...), one lane per vector
// (its tensor-memory lane): the norm n = ||x|| from the vector's bf16 row in the
// ring, then y = (Pi x) / n in chunks of 32 columns through the same cell-table
// quantizer, pair table and packing as the FWHT kernels.
constexpr int kGM = 128;                      // vectors per tile (MMA M)
constexpr int kGStages = 3;                   // X tiles in the ring
constexpr int kGAcc = 4;                      // accumulators (4 x 128 = 512 tensor-memory columns)
constexpr int kGWarps = 2 + 4 * kGAcc;        // copy warp, MMA warp, 4 epilogue warps per accumulator
constexpr uint32_t kGTile = kGM * kD * 2;     // 32 KB of bf16 vectors
constexpr uint32_t kGMat = kD * kD * 2;       // 32 KB: one bf16 part of Pi
// from the 16 KB aligned base: cell table 16 KB, pair table 32 KB, barriers 1 KB,
// Pi parts 64 KB, ring 96 KB (every matrix 1 KB aligned)
constexpr uint32_t kGOffPair = 16384, kGOffMisc = 49152, kGOffPi = 50176, kGOffX = kGOffPi + 2 * kGMat;
constexpr size_t kGSmem = 16384 + (size_t)kGOffX + (size_t)kGStages * kGTile;

struct QuantGemmArgs {
  CUtensorMap tm[2];  // [n_vec][128] bf16 keys / values: box [128][64], 128-byte swizzle
  uint8_t* pool[2];
  const int64_t* slots;
  int tiles;          // 128-vector tiles per tensor
  uint32_t n_vec;     // vectors per tensor
  int ny;
  int H;
  int page_bytes;
  int64_t max_slot;
  const float* rot;   // Pi [128][128] row-major (y = Pi x)
  Codebook cb;
  int norm_mode;
  unsigned* status;
};

template <int BITS>
__global__ void __launch_bounds__(kGWarps * 32, 1) k_quantize_dense_mma(const __grid_constant__ QuantGemmArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent decode may start its prologue
  constexpr int R = 16 * BITS;
  constexpr uint32_t kIdesc = umma_idesc_bf16_f32(kGM, kD);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const uint32_t A0 = (sbase + 16383u) & ~16383u;
  const uint32_t cell_addr = A0, pair_addr = A0 + kGOffPair, misc_addr = A0 + kGOffMisc;
  const uint32_t pi_addr = A0 + kGOffPi, x_addr = A0 + kGOffX;
  auto gen = [&](uint32_t addr) { return smem_raw + (addr - sbase); };
  uint64_t* full = reinterpret_cast<uint64_t*>(gen(misc_addr));  // [kGStages] X tile landed
  uint64_t* empty = full + kGStages;                              // [kGStages] MMAs and norms done with it
  uint64_t* mdone = empty + kGStages;                             // [kGAcc] accumulator written
  uint64_t* aempty = mdone + kGAcc;                               // [kGAcc] accumulator read out
  const uint32_t tmem_slot = misc_addr + 512;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = a.tiles * a.ny;
  const int n_my = (int)blockIdx.x < total ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1 + 4);  // the MMA commit and the 4 epilogue warps of the tile
    }
    for (int e = 0; e < kGAcc; ++e) {
      mbar_init(mdone + e, 1);
      mbar_init(aempty + e, 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);

  build_pair_cell_tables<BITS>(a.cb, gen(cell_addr), gen(pair_addr));
  // Pi -> bf16 parts, element (n = i, k = j) of B = Pi at box j / 64, row i, chunk (j % 64) / 8 ^ (i & 7);
  // each thread's loads in flight together
  constexpr int kPiIters = (kD * kD / 8 + kGWarps * 32 - 1) / (kGWarps * 32);
  float4 pl[kPiIters][2];
#pragma unroll
  for (int it = 0; it < kPiIters; ++it) {
    const int c = (int)threadIdx.x + it * kGWarps * 32;
    if (c < kD * kD / 8) {
      pl[it][0] = __ldg(reinterpret_cast<const float4*>(a.rot) + 2 * c);
      pl[it][1] = __ldg(reinterpret_cast<const float4*>(a.rot) + 2 * c + 1);
    }
  }
#pragma unroll
  for (int it = 0; it < kPiIters; ++it) {
    const int c = (int)threadIdx.x + it * kGWarps * 32;
    if (c >= kD * kD / 8) break;
    const int i = c >> 4, kc = c & 15;
    const float4 p0 = pl[it][0], p1 = pl[it][1];
    const float v[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]), h1 = __float2bfloat16_rn(v[2 * e + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
      hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    const uint32_t off = (uint32_t)(kc >> 3) * (kGMat / 2) + (uint32_t)i * 128u + ((uint32_t)((kc & 7) ^ (i & 7)) << 4);
    *reinterpret_cast<uint4*>(gen(pi_addr + off)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(gen(pi_addr + kGMat + off)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  fence_proxy_async();  // Pi parts (generic stores) are read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gen(tmem_slot));

  if (warp == 0) {
    if (lane == 0) {  // copies: tile i of this CTA into stage i % kGStages
      int issued = 0;
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kGStages;
        if (i >= kGStages && !mbar_wait(empty + s, (uint32_t)((i / kGStages) - 1) & 1u)) {
          flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
          break;
        }
        const int tile = (int)blockIdx.x + i * (int)gridDim.x;
        const int kv = tile >= a.tiles ? 1 : 0;
        const int row = (tile - kv * a.tiles) * kGM;
        mbar_arrive_expect_tx(full + s, kGTile);
        tensor_copy_2d(x_addr + (uint32_t)s * kGTile, &a.tm[kv], 0, row, full + s);
        tensor_copy_2d(x_addr + (uint32_t)s * kGTile + kGTile / 2, &a.tm[kv], 64, row, full + s);
        issued = i + 1;
      }
      // copies still in flight land before the CTA can exit (all of them on the normal path)
      for (int i = issued - kGStages < 0 ? 0 : issued - kGStages; i < issued; ++i)
        mbar_wait(full + i % kGStages, (uint32_t)(i / kGStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMAs of tile i into accumulator i % kGAcc
      int issued = 0;
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kGStages, e = i % kGAcc;
        if (!mbar_wait(full + s, (uint32_t)(i / kGStages) & 1u) ||
            (i >= kGAcc && !mbar_wait(aempty + e, (uint32_t)((i / kGAcc) - 1) & 1u))) {
          flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)e * kD;
        const uint32_t xs = x_addr + (uint32_t)s * kGTile;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {  // K step of 16: box kc / 4, 32 bytes into the swizzled rows
          const uint32_t ko = (uint32_t)(kc >> 2) * (kGTile / 2) + (uint32_t)(kc & 3) * 32u;
          const uint32_t po = (uint32_t)(kc >> 2) * (kGMat / 2) + (uint32_t)(kc & 3) * 32u;
          const uint64_t ad = umma_desc_sw128(xs + ko);
          umma_bf16(d, ad, umma_desc_sw128(pi_addr + po), kIdesc, kc > 0);
          umma_bf16(d, ad, umma_desc_sw128(pi_addr + kGMat + po), kIdesc, true);
        }
        umma_commit(smem_u32(empty + s));
        umma_commit(smem_u32(mdone + e));
        issued = i + 1;
      }
      if (issued > 0)  // every MMA has completed before tensor memory is released
        mbar_wait(mdone + (issued - 1) % kGAcc, (uint32_t)((issued - 1) / kGAcc) & 1u);
    }
  } else {
    const int grp = (warp - 2) >> 2;           // accumulator served
    const int quad = warp & 3;                 // tensor-memory lanes 32 quad .. 32 quad + 31
    const int r = quad * 32 + lane;            // row of the tile
    const uint32_t qrow = cell_addr | ((uint32_t)(lane & 15) << 3);
    const uint32_t prow = pair_addr + ((uint32_t)lane << 2);
    const uint32_t xrow = x_addr + (uint32_t)r * 128u + ((uint32_t)(r & 7) << 4);  // with the swizzle bits
    for (int i = grp; i < n_my; i += kGAcc) {
      const int s = i % kGStages;
      const int tile = (int)blockIdx.x + i * (int)gridDim.x;
      const int kv = tile >= a.tiles ? 1 : 0;
      const uint32_t vec = (uint32_t)((tile - kv * a.tiles) * kGM + r);
      const bool valid = vec < a.n_vec;
      const uint32_t tok = valid ? vec / (uint32_t)a.H : 0u;
      const int head = (int)(vec - tok * (uint32_t)a.H);
      const int64_t slot = valid ? __ldg(a.slots + tok) : -1;
      // the accumulator first: its MMAs consumed phase i / kGStages of full[s], so that
      // phase is complete (and the next cannot start before this warp arrives on empty[s])
      if (!mbar_wait(mdone + grp, (uint32_t)(i / kGAcc) & 1u) || !mbar_wait(full + s, (uint32_t)(i / kGStages) & 1u)) {
        if (lane == 0) flag_status(a.status, TQ_DEV_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      // n = ||x|| from the bf16 row
      const uint32_t xb = xrow + (uint32_t)s * kGTile;
      float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 d0 = lds128u(xb ^ ((uint32_t)c << 4));
        const uint4 d1 = lds128u((xb + kGTile / 2) ^ ((uint32_t)c << 4));
        const uint32_t w[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 p = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
          ss2 = __ffma2_rn(p, p, ss2);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);  // this warp is done with the X tile
      const float n = sqrtf(ss2.x + ss2.y);
      const float inv_n = n > 0.0f ? 1.0f / n : 0.0f;
      const float2 s2 = make_float2(inv_n, inv_n);

      uint32_t wd[4 * BITS];
      float2 c2p = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {  // coordinates 32 ch .. 32 ch + 31
        float y[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)grp * kD + (uint32_t)ch * 32u, y);
        uint32_t wc[BITS];
        cell_chunk32<BITS>(y, s2, qrow, prow, wc, c2p);
#pragma unroll
        for (int k = 0; k < BITS; ++k) wd[ch * BITS + k] = wc[k];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty + grp);  // accumulator read out

      const float c2 = c2p.x + c2p.y;
      float gamma;
      if (a.norm_mode == TQ_NORM_RAW) gamma = n;
      else gamma = (n > 0.0f && c2 > 0.0f) ? n / sqrtf(c2) : 0.0f;
      if (valid && slot >= a.max_slot) {
        flag_status(a.status, TQ_DEV_BAD_SLOT);
      } else if (valid && slot >= 0) {
        uint8_t* page = a.pool[kv] + ((slot >> 4) * a.H + head) * (int64_t)a.page_bytes;
        const int off = (int)(slot & 15);
        uint4* rec = reinterpret_cast<uint4*>(page + off * R);
#pragma unroll
        for (int k = 0; k < BITS; ++k) rec[k] = make_uint4(wd[4 * k], wd[4 * k + 1], wd[4 * k + 2], wd[4 * k + 3]);
        *reinterpret_cast<float*>(page + 16 * R + 4 * off) = gamma;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  grid_dep_wait();  // complete only after a grid this one is a programmatic dependent of
}

// The quantizer of the two bulk append kernels on given rotated coordinates:
// tq_quantize_rotated runs it whenever a bf16 append of the same layer and size
// would run k_quantize_tma (SPLIT: Hadamard layers, at least kTmaMinVectors
// vectors) or k_quantize_dense_mma (!SPLIT: dense layers), so that those
// kernels' cell-table quantizer, pair-table norm and packing can be checked on
// exact inputs.  One lane per vector; y is read from global memory in the
// layout the bulk kernel holds it in registers.  y is clamped to [-1, 1] before
// the lookup, which changes no code (every boundary lies inside (-1, 1)) and
// keeps the cell index in range for any input.
__device__ __forceinline__ float clamp_unit(float y) { return fminf(fmaxf(y, -1.0f), 1.0f); }

constexpr size_t kCellSmem = 16384 + kTCellBytes + kTPairBytes;

template <int BITS, bool SPLIT>
__global__ void __launch_bounds__(256) k_quantize_given_y_cells(QuantArgs a) {
  constexpr int R = 16 * BITS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  const uint32_t cell_addr = (sbase + 16383u) & ~16383u;  // 16 KB aligned: address = (t & mask) | row
  const uint32_t pair_addr = cell_addr + kTCellBytes;
  build_pair_cell_tables<BITS>(a.cb, smem_raw + (cell_addr - sbase), smem_raw + (pair_addr - sbase));
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint32_t qrow = cell_addr | ((uint32_t)(lane & 15) << 3);
  const uint32_t prow = pair_addr + ((uint32_t)lane << 2);
  const float2 one = make_float2(1.0f, 1.0f);
  for (int64_t vec = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; vec < a.n_vec;
       vec += (int64_t)gridDim.x * blockDim.x) {
    const float* yr = a.y + vec * kD;
    const float n = __ldg(a.norms + vec);
    uint32_t wd[4 * BITS];
    float c2;
    if constexpr (SPLIT) {
      float2 v[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] = make_float2(clamp_unit(__ldg(yr + j)), clamp_unit(__ldg(yr + 64 + j)));
      c2 = cell_record_split<BITS>(v, one, qrow, prow, wd);
    } else {
      float2 c2p = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = clamp_unit(__ldg(yr + 32 * ch + j));
        uint32_t wc[BITS];
        cell_chunk32<BITS>(y, one, qrow, prow, wc, c2p);
#pragma unroll
        for (int k = 0; k < BITS; ++k) wd[ch * BITS + k] = wc[k];
      }
      c2 = c2p.x + c2p.y;
    }
    float gamma;
    if (a.norm_mode == TQ_NORM_RAW) gamma = n;
    else gamma = (n > 0.0f && c2 > 0.0f) ? n / sqrtf(c2) : 0.0f;
    const int64_t tok = vec / a.H;
    const int head = (int)(vec - tok * a.H);
    const int64_t slot = __ldg(a.slots + tok);
    if (slot >= a.max_slot) {
      flag_status(a.status, TQ_DEV_BAD_SLOT);
    } else if (slot >= 0) {
      uint8_t* page = a.pool + ((slot >> 4) * a.H + head) * (int64_t)a.page_bytes;
      const int off = (int)(slot & 15);
      uint4* rec = reinterpret_cast<uint4*>(page + off * R);
#pragma unroll
      for (int k = 0; k < BITS; ++k) rec[k] = make_uint4(wd[4 * k], wd[4 * k + 1], wd[4 * k + 2], wd[4 * k + 3]);
      *reinterpret_cast<float*>(page + 16 * R + 4 * off) = gamma;
    }
  }
}

// bf16 layers: the append is a paged copy with rounding to bf16.
template <typename TIn>
__global__ void __launch_bounds__(256) k_append_bf16(const TIn* __restrict__ x, const int64_t* __restrict__ slots,
                                                     int64_t n_vec, int H, int64_t max_slot, uint8_t* pool,
                                                     unsigned* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent decode may start its prologue
  const int64_t n_chunks = n_vec * 16;  // 8 elements per chunk
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n_chunks; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t vec = c >> 4;
    const int part = (int)(c & 15);
    const int64_t tok = vec / H;
    const int head = (int)(vec - tok * H);
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0) continue;
    if (slot >= max_slot) {
      if (part == 0) flag_status(status, TQ_DEV_BAD_SLOT);
      continue;
    }
    const TIn* src = x + vec * kD + part * 8;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat16 lo = __float2bfloat16_rn(load_elem<TIn>(src + 2 * k));
      const __nv_bfloat16 hi = __float2bfloat16_rn(load_elem<TIn>(src + 2 * k + 1));
      w[k] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    uint8_t* page = pool + ((slot >> 4) * H + head) * (int64_t)(kBlock * kD * 2);
    *reinterpret_cast<uint4*>(page + (slot & 15) * (kD * 2) + part * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// k8v4 keys: each coordinate as FP8 E4M3 (nearest, ties to even, saturating at
// +-448), 128-byte records, 16 per (block, KV head) page.  One thread per 16
// coordinates (one 16-byte store).
template <typename TIn>
__global__ void __launch_bounds__(256) k_append_fp8(const TIn* __restrict__ x, const int64_t* __restrict__ slots,
                                                    int64_t n_vec, int H, int64_t max_slot, uint8_t* pool,
                                                    unsigned* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent decode may start its prologue
  const int64_t n_chunks = n_vec * 8;  // 16 coordinates per chunk
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n_chunks; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t vec = c >> 3;
    const int part = (int)(c & 7);
    const int64_t tok = vec / H;
    const int head = (int)(vec - tok * H);
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0) continue;
    if (slot >= max_slot) {
      if (part == 0) flag_status(status, TQ_DEV_BAD_SLOT);
      continue;
    }
    const TIn* src = x + vec * kD + part * 16;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(load_elem<TIn>(src + 4 * k), load_elem<TIn>(src + 4 * k + 1)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(load_elem<TIn>(src + 4 * k + 2), load_elem<TIn>(src + 4 * k + 3)), __NV_SATFINITE, __NV_E4M3);
      w[k] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    uint8_t* page = pool + ((slot >> 4) * H + head) * (int64_t)(kBlock * kD);
    *reinterpret_cast<uint4*>(page + (slot & 15) * kD + part * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <typename TOut>
__global__ void __launch_bounds__(256) k_dequant_fp8(const uint8_t* __restrict__ pool, int H, int64_t max_slot,
                                                     const int64_t* __restrict__ slots, int64_t n_vec, TOut* out,
                                                     unsigned* status) {
  const int64_t n = n_vec * kD;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t vec = e / kD;
    const int j = (int)(e - vec * kD);
    const int64_t tok = vec / H;
    const int head = (int)(vec - tok * H);
    const int64_t slot = __ldg(slots + tok);
    float v = 0.0f;
    if (slot >= 0 && slot < max_slot) {
      const uint8_t b = pool[((slot >> 4) * H + head) * (int64_t)(kBlock * kD) + (slot & 15) * kD + j];
      v = __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
    } else if (slot >= max_slot && j == 0) {
      flag_status(status, TQ_DEV_BAD_SLOT);
    }
    store_elem<TOut>(out + e, v);
  }
}

// Dequantize: x_hat = gamma Pi^T c[idx] (rotated-domain values, then the inverse rotation).
template <int BITS, typename TOut, bool DENSE>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t* __restrict__ pool, int page_bytes, int H,
                                                    int64_t max_slot, const int64_t* __restrict__ slots, int64_t n_vec,
                                                    const float* __restrict__ rot, Codebook cb, TOut* out,
                                                    unsigned* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int R = 16 * BITS;
  uint32_t* signw = reinterpret_cast<uint32_t*>(smem_raw);
  float* ctab = reinterpret_cast<float*>(smem_raw + 16);  // [16][32]
  float* tile = reinterpret_cast<float*>(smem_raw + kTableBytes);
  float* matP = reinterpret_cast<float*>(smem_raw + kTableBytes + kTileBytes);
  const int tid = threadIdx.x, lane = tid & 31, q = tid & 3, vl = tid >> 2;
  for (int i = tid; i < 16 * 32; i += kThreads) ctab[i] = cb.c[(i / 32) & ((1 << BITS) - 1)];
  if (!DENSE && tid < 32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t m = __ballot_sync(0xffffffffu, __ldg(rot + 32 * k + lane) < 0.0f);
      if (lane == 0) signw[k] = m;
    }
  }
  if (DENSE) stage_matrix(rot, matP, /*transpose=*/false);  // out = Pi^T v
  __syncthreads();
  const uint32_t sw = DENSE ? 0u : signw[q];
  const int64_t n_tiles = (n_vec + kTile - 1) / kTile;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t vec_raw = t * kTile + vl;
    const bool valid = vec_raw < n_vec;
    const int64_t vec = valid ? vec_raw : (n_vec - 1);
    const int64_t tok = vec / H;
    const int head = (int)(vec - tok * H);
    const int64_t slot = __ldg(slots + tok);
    const bool ok = slot >= 0 && slot < max_slot;
    if (valid && slot >= max_slot && q == 0) flag_status(status, TQ_DEV_BAD_SLOT);
    float v[32];
    if (ok) {
      const uint8_t* page = pool + ((slot >> 4) * H + head) * (int64_t)page_bytes;
      const uint32_t* rec = reinterpret_cast<const uint32_t*>(page + (slot & 15) * R + 4 * BITS * q);
      uint32_t w[BITS + 1];
#pragma unroll
      for (int i = 0; i < BITS; ++i) w[i] = rec[i];
      w[BITS] = 0u;
      const float gamma = *reinterpret_cast<const float*>(page + 16 * R + 4 * (slot & 15));
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int bit = BITS * k;
        uint32_t c = w[bit >> 5] >> (bit & 31);
        if ((bit & 31) + BITS > 32) c |= w[(bit >> 5) + 1] << (32 - (bit & 31));
        c &= (1u << BITS) - 1u;
        v[k] = gamma * ctab[c * 32 + lane];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = 0.0f;
    }
    if constexpr (DENSE) {
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 32; ++i) tile[vl * kTileStride + 32 * q + i] = v[i];
      __syncthreads();
      matvec_padded(matP, tile + vl * kTileStride, q, v);
    } else {
      fwht128_quad(v, q);  // Pi^T v = D H v / sqrt(d)
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = flip_sign(v[i] * 0.08838834764831845f, sw, i);
    }
    if (valid) {
      TOut* o = out + vec * kD + 32 * q;
#pragma unroll
      for (int i = 0; i < 32; ++i) store_elem<TOut>(o + i, v[i]);
    }
  }
}

template <typename TOut>
__global__ void __launch_bounds__(256) k_dequant_bf16(const uint8_t* __restrict__ pool, int H, int64_t max_slot,
                                                      const int64_t* __restrict__ slots, int64_t n_vec, TOut* out,
                                                      unsigned* status) {
  const int64_t n = n_vec * kD;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t vec = e / kD;
    const int j = (int)(e - vec * kD);
    const int64_t tok = vec / H;
    const int head = (int)(vec - tok * H);
    const int64_t slot = __ldg(slots + tok);
    float v = 0.0f;
    if (slot >= 0 && slot < max_slot) {
      const uint16_t* page =
          reinterpret_cast<const uint16_t*>(pool + ((slot >> 4) * H + head) * (int64_t)(kBlock * kD * 2));
      v = bf16_bits_to_float(page[(slot & 15) * kD + j]);
    } else if (slot >= max_slot && j == 0) {
      flag_status(status, TQ_DEV_BAD_SLOT);
    }
    store_elem<TOut>(out + e, v);
  }
}

// ----------------------------------------------------------------- launchers

Codebook codebook_of(const tq_cache_desc& d, int which) {
  Codebook cb;
  const float* c = which == 0 ? d.centroids_k : d.centroids_v;
  const float* b = which == 0 ? d.boundaries_k : d.boundaries_v;
  for (int i = 0; i < 16; ++i) cb.c[i] = c[i];
  for (int i = 0; i < 15; ++i) cb.b[i] = b[i];
  return cb;
}

template <int BITS, typename TIn, int MODE, bool QJL>
static cudaError_t run_quantize(const QuantArgs& a, int ny, int num_sms, cudaStream_t st) {
  auto kern = k_quantize<BITS, TIn, MODE, QJL>;
  size_t smem = kTableBytes;
  if (MODE != MODE_GIVEN_Y) smem += 16384 + kLutQBytes;  // the cell table is 16 KB aligned
  if (MODE == MODE_DENSE || QJL) smem += kTileBytes;
  if (MODE == MODE_DENSE) smem += kMatBytes;
  if (QJL) smem += kMatBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.n_vec + kTile - 1) / kTile;
  const int per_sm = (MODE == MODE_DENSE || QJL) ? 1 : 8;
  const int64_t cap = (int64_t)num_sms * per_sm / ny;
  int64_t grid = tiles < cap ? tiles : cap;
  if (grid < 1) grid = 1;
  kern<<<dim3((unsigned)grid, (unsigned)ny), kThreads, smem, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS, typename TIn>
static cudaError_t dispatch_mode(const QuantArgs& a, int ny, int mode, bool qjl, int num_sms, cudaStream_t st) {
  if (mode == MODE_GIVEN_Y) return run_quantize<BITS, float, MODE_GIVEN_Y, false>(a, ny, num_sms, st);
  if (mode == MODE_HADAMARD)
    return qjl ? run_quantize<BITS, TIn, MODE_HADAMARD, true>(a, ny, num_sms, st)
               : run_quantize<BITS, TIn, MODE_HADAMARD, false>(a, ny, num_sms, st);
  return qjl ? run_quantize<BITS, TIn, MODE_DENSE, true>(a, ny, num_sms, st)
             : run_quantize<BITS, TIn, MODE_DENSE, false>(a, ny, num_sms, st);
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link-time libcuda dependency).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [n_vec][128] bf16 rows, boxes of [box_rows rows][64 elements] with the 128-byte swizzle.
static bool vec_tensor_map(CUtensorMap* m, const void* x, uint32_t n_vec, uint32_t box_rows) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)n_vec};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches kern<<<grid, block, smem, st>>>(args); with pdl, as a programmatic dependent
// of the kernel before it on the stream (it may start while that kernel finishes).
template <typename Args>
static cudaError_t launch_maybe_pdl(void (*kern)(Args), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                                    const Args& args, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BITS>
static cudaError_t run_quantize_tma(const QuantTmaArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  auto kern = k_quantize_tma<BITS>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTSmem);
  if (e != cudaSuccess) return e;
  const int64_t total = a.tiles * a.ny;
  int64_t grid = (total + kTW - 1) / kTW;
  if (grid > num_sms) grid = num_sms;
  return launch_maybe_pdl(kern, (unsigned)grid, kTW * 32, kTSmem, st, a, pdl);
}

// The staged kernel takes bf16 Hadamard appends without QJL whose inputs TMA can
// address (16-byte aligned, fewer than 2^31 vectors) and that are large enough
// to amortise its per-CTA tables (at least kTmaMinVectors vectors in the launch;
// a decode step's append of a few tokens is faster on the plain kernel).
// Returns false (nothing launched) when the append is not of that kind.
constexpr int64_t kTmaMinVectors = 24576;
static bool try_quantize_tma(const tq_cache_desc& d, int which, const void* x, const void* x_v, int bits,
                             const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms, cudaStream_t st,
                             cudaError_t* err, bool pdl) {
  const int64_t n_vec = n_tok * d.num_kv_heads;
  if (n_vec <= 0 || n_vec >= ((int64_t)1 << 31)) return false;
  if (n_vec * (x_v ? 2 : 1) < kTmaMinVectors) return false;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (x_v && (reinterpret_cast<uintptr_t>(x_v) & 15u))) return false;
  QuantTmaArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!vec_tensor_map(&a.tm[0], x, (uint32_t)n_vec, 32)) return false;
  if (x_v && !vec_tensor_map(&a.tm[1], x_v, (uint32_t)n_vec, 32)) return false;
  a.pool[0] = reinterpret_cast<uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  a.pool[1] = reinterpret_cast<uint8_t*>(d.v_cache);
  a.slots = slots;
  a.tiles = (n_vec + 31) / 32;
  a.n_vec = (uint32_t)n_vec;
  a.ny = x_v ? 2 : 1;
  a.H = d.num_kv_heads;
  a.page_bytes = (int)page_bytes_of(d, which);
  a.max_slot = d.num_blocks * kBlock;
  a.rot = d.rotation;
  a.cb = codebook_of(d, which);
  a.norm_mode = d.fmt.norm_mode;
  a.status = status;
  switch (bits) {
    case 2: *err = run_quantize_tma<2>(a, num_sms, st, pdl); break;
    case 3: *err = run_quantize_tma<3>(a, num_sms, st, pdl); break;
    default: *err = run_quantize_tma<4>(a, num_sms, st, pdl); break;
  }
  return true;
}

template <int BITS>
static cudaError_t run_quantize_dense_mma(const QuantGemmArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  auto kern = k_quantize_dense_mma<BITS>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
  if (e != cudaSuccess) return e;
  const int total = a.tiles * a.ny;
  const int grid = total < num_sms ? total : num_sms;
  return launch_maybe_pdl(kern, (unsigned)grid, kGWarps * 32, kGSmem, st, a, pdl);
}

// bf16 appends through a dense Pi without QJL go to the tensor-core kernel (TMA
// addressable inputs, fewer than 2^31 vectors); it is also the faster one for a
// decode step's few tokens.  Returns false (nothing launched) for other appends.
static bool try_quantize_dense_mma(const tq_cache_desc& d, int which, const void* x, const void* x_v, int bits,
                                   const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms,
                                   cudaStream_t st, cudaError_t* err, bool pdl) {
  const int64_t n_vec = n_tok * d.num_kv_heads;
  if (n_vec <= 0 || n_vec >= ((int64_t)1 << 31) - kGM) return false;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (x_v && (reinterpret_cast<uintptr_t>(x_v) & 15u))) return false;
  if (reinterpret_cast<uintptr_t>(d.rotation) & 15u) return false;
  QuantGemmArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!vec_tensor_map(&a.tm[0], x, (uint32_t)n_vec, kGM)) return false;
  if (x_v && !vec_tensor_map(&a.tm[1], x_v, (uint32_t)n_vec, kGM)) return false;
  a.pool[0] = reinterpret_cast<uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  a.pool[1] = reinterpret_cast<uint8_t*>(d.v_cache);
  a.slots = slots;
  a.tiles = (int)((n_vec + kGM - 1) / kGM);
  a.n_vec = (uint32_t)n_vec;
  a.ny = x_v ? 2 : 1;
  a.H = d.num_kv_heads;
  a.page_bytes = (int)page_bytes_of(d, which);
  a.max_slot = d.num_blocks * kBlock;
  a.rot = d.rotation;
  a.cb = codebook_of(d, which);
  a.norm_mode = d.fmt.norm_mode;
  a.status = status;
  switch (bits) {
    case 2: *err = run_quantize_dense_mma<2>(a, num_sms, st, pdl); break;
    case 3: *err = run_quantize_dense_mma<3>(a, num_sms, st, pdl); break;
    default: *err = run_quantize_dense_mma<4>(a, num_sms, st, pdl); break;
  }
  return true;
}

template <int BITS, bool SPLIT>
static cudaError_t run_given_y_cells(const QuantArgs& a, int num_sms, cudaStream_t st) {
  auto kern = k_quantize_given_y_cells<BITS, SPLIT>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCellSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = (a.n_vec + 255) / 256;
  if (grid > (int64_t)num_sms * 3) grid = (int64_t)num_sms * 3;
  kern<<<(unsigned)grid, 256, kCellSmem, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

static QuantArgs quant_args(const tq_cache_desc& d, int which, const void* x, const float* y, const float* norms,
                            const int64_t* slots, int64_t n_tok, unsigned* status) {
  QuantArgs a;
  a.x = x;
  a.y = y;
  a.norms = norms;
  a.slots = slots;
  a.n_vec = n_tok * d.num_kv_heads;
  a.H = d.num_kv_heads;
  a.max_slot = d.num_blocks * kBlock;
  a.pool = reinterpret_cast<uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  a.page_bytes = (int)page_bytes_of(d, which);
  a.rot = d.rotation;
  a.qjl = d.qjl_proj;
  a.cb = codebook_of(d, which);
  a.norm_mode = d.fmt.norm_mode;
  a.status = status;
  a.x_v = nullptr;
  a.pool_v = nullptr;
  return a;
}

cudaError_t launch_quantize(const tq_cache_desc& d, int which, const void* x, int in_dtype, const float* y,
                            const float* norms, const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms,
                            cudaStream_t st, const void* x_v, bool pdl) {
  if (n_tok <= 0) return cudaSuccess;
  if (d.fmt.kv_format == TQ_KV_POLAR) return launch_polar_append(d, which, x, in_dtype, slots, n_tok, status, num_sms, st);
  const int64_t n_vec = n_tok * d.num_kv_heads;
  const int64_t max_slot = d.num_blocks * kBlock;
  uint8_t* pool = reinterpret_cast<uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  if (d.fmt.kv_format == TQ_KV_K8V4 && which == 0) {  // FP8 keys
    int64_t grid = (n_vec * 8 + 255) / 256;
    if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
    if (in_dtype == TQ_F32)
      k_append_fp8<float><<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const float*>(x), slots, n_vec,
                                                          d.num_kv_heads, max_slot, pool, status);
    else
      k_append_fp8<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), slots,
                                                                  n_vec, d.num_kv_heads, max_slot, pool, status);
    count_launch();
    return cudaGetLastError();
  }
  if (d.fmt.kv_format == TQ_KV_BF16) {
    int64_t chunks = n_vec * 16;
    int64_t grid = (chunks + 255) / 256;
    if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
    if (in_dtype == TQ_F32)
      k_append_bf16<float><<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const float*>(x), slots, n_vec,
                                                           d.num_kv_heads, max_slot, pool, status);
    else
      k_append_bf16<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), slots,
                                                                   n_vec, d.num_kv_heads, max_slot, pool, status);
    count_launch();
    return cudaGetLastError();
  }
  const int bits = which == 0 ? d.fmt.bits_k : d.fmt.bits_v;
  const bool qjl = which == 0 && d.fmt.qjl_k && y == nullptr;
  const int mode = y ? MODE_GIVEN_Y : (d.fmt.rot_kind == TQ_ROT_DENSE ? MODE_DENSE : MODE_HADAMARD);
  if (mode == MODE_GIVEN_Y && (d.fmt.rot_kind == TQ_ROT_DENSE || n_vec >= kTmaMinVectors)) {
    const QuantArgs a = quant_args(d, which, nullptr, y, norms, slots, n_tok, status);
    const bool split = d.fmt.rot_kind != TQ_ROT_DENSE;
    switch (bits) {
      case 2: return split ? run_given_y_cells<2, true>(a, num_sms, st) : run_given_y_cells<2, false>(a, num_sms, st);
      case 3: return split ? run_given_y_cells<3, true>(a, num_sms, st) : run_given_y_cells<3, false>(a, num_sms, st);
      default: return split ? run_given_y_cells<4, true>(a, num_sms, st) : run_given_y_cells<4, false>(a, num_sms, st);
    }
  }
  if (mode == MODE_HADAMARD && !qjl && in_dtype == TQ_BF16) {
    cudaError_t err = cudaSuccess;
    if (try_quantize_tma(d, which, x, x_v, bits, slots, n_tok, status, num_sms, st, &err, pdl)) return err;
  }
  if (mode == MODE_DENSE && !qjl && in_dtype == TQ_BF16) {
    cudaError_t err = cudaSuccess;
    if (try_quantize_dense_mma(d, which, x, x_v, bits, slots, n_tok, status, num_sms, st, &err, pdl)) return err;
  }
  QuantArgs a = quant_args(d, which, x, y, norms, slots, n_tok, status);
  int ny = 1;
  if (x_v) {  // values in the same launch (caller checked that the formats and tables agree)
    a.x_v = x_v;
    a.pool_v = reinterpret_cast<uint8_t*>(d.v_cache);
    ny = 2;
  }
  const bool f32 = in_dtype == TQ_F32;
  switch (bits) {
    case 2:
      return f32 ? dispatch_mode<2, float>(a, ny, mode, qjl, num_sms, st)
                 : dispatch_mode<2, __nv_bfloat16>(a, ny, mode, qjl, num_sms, st);
    case 3:
      return f32 ? dispatch_mode<3, float>(a, ny, mode, qjl, num_sms, st)
                 : dispatch_mode<3, __nv_bfloat16>(a, ny, mode, qjl, num_sms, st);
    default:
      return f32 ? dispatch_mode<4, float>(a, ny, mode, qjl, num_sms, st)
                 : dispatch_mode<4, __nv_bfloat16>(a, ny, mode, qjl, num_sms, st);
  }
}

template <int BITS, typename TOut, bool DENSE>
static cudaError_t run_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n_vec, void* out,
                               unsigned* status, int num_sms, cudaStream_t st) {
  auto kern = k_dequant<BITS, TOut, DENSE>;
  size_t smem = kTableBytes + (DENSE ? kTileBytes + kMatBytes : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (n_vec + kTile - 1) / kTile;
  int64_t grid = tiles < (int64_t)num_sms * 4 ? tiles : (int64_t)num_sms * 4;
  if (grid < 1) grid = 1;
  const uint8_t* pool = reinterpret_cast<const uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
  kern<<<(unsigned)grid, kThreads, smem, st>>>(pool, (int)page_bytes_of(d, which), d.num_kv_heads,
                                              d.num_blocks * kBlock, slots, n_vec, d.rotation, codebook_of(d, which),
                                              reinterpret_cast<TOut*>(out), status);
  count_launch();
  return cudaGetLastError();
}

template <typename TOut>
static cudaError_t dequant_bits(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n_vec, void* out,
                                unsigned* status, int num_sms, cudaStream_t st) {
  const int bits = which == 0 ? d.fmt.bits_k : d.fmt.bits_v;
  const bool dense = d.fmt.rot_kind == TQ_ROT_DENSE;
  switch (bits) {
    case 2:
      return dense ? run_dequant<2, TOut, true>(d, which, slots, n_vec, out, status, num_sms, st)
                   : run_dequant<2, TOut, false>(d, which, slots, n_vec, out, status, num_sms, st);
    case 3:
      return dense ? run_dequant<3, TOut, true>(d, which, slots, n_vec, out, status, num_sms, st)
                   : run_dequant<3, TOut, false>(d, which, slots, n_vec, out, status, num_sms, st);
    default:
      return dense ? run_dequant<4, TOut, true>(d, which, slots, n_vec, out, status, num_sms, st)
                   : run_dequant<4, TOut, false>(d, which, slots, n_vec, out, status, num_sms, st);
  }
}

cudaError_t launch_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n, void* out,
                           int out_dtype, unsigned* status, int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (d.fmt.kv_format == TQ_KV_POLAR) return launch_polar_dequant(d, which, slots, n, out, out_dtype, status, num_sms, st);
  const int64_t n_vec = n * d.num_kv_heads;
  if (d.fmt.kv_format == TQ_KV_K8V4 && which == 0) {
    const uint8_t* pool = reinterpret_cast<const uint8_t*>(d.k_cache);
    int64_t grid = (n_vec * kD + 255) / 256;
    if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
    if (out_dtype == TQ_F32)
      k_dequant_fp8<float><<<(unsigned)grid, 256, 0, st>>>(pool, d.num_kv_heads, d.num_blocks * kBlock, slots, n_vec,
                                                          reinterpret_cast<float*>(out), status);
    else
      k_dequant_fp8<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(pool, d.num_kv_heads, d.num_blocks * kBlock, slots,
                                                                  n_vec, reinterpret_cast<__nv_bfloat16*>(out),
                                                                  status);
    count_launch();
    return cudaGetLastError();
  }
  if (d.fmt.kv_format == TQ_KV_BF16) {
    const uint8_t* pool = reinterpret_cast<const uint8_t*>(which == 0 ? d.k_cache : d.v_cache);
    int64_t grid = (n_vec * kD + 255) / 256;
    if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
    if (out_dtype == TQ_F32)
      k_dequant_bf16<float><<<(unsigned)grid, 256, 0, st>>>(pool, d.num_kv_heads, d.num_blocks * kBlock, slots, n_vec,
                                                             reinterpret_cast<float*>(out), status);
    else
      k_dequant_bf16<__nv_bfloat16><<<(unsigned)grid, 256, 0, st>>>(pool, d.num_kv_heads, d.num_blocks * kBlock,
                                                                     slots, n_vec,
                                                                     reinterpret_cast<__nv_bfloat16*>(out), status);
    count_launch();
    return cudaGetLastError();
  }
  return out_dtype == TQ_F32 ? dequant_bits<float>(d, which, slots, n_vec, out, status, num_sms, st)
                             : dequant_bits<__nv_bfloat16>(d, which, slots, n_vec, out, status, num_sms, st);
}

}  // namespace tq
