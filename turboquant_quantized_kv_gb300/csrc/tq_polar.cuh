// Device code of the PolarQuant-variant layers shared by tq_polar.cu (append,
// dequantize, combine, launch) and the decode translation units
// tq_polar_decode_k{2,3,4}.cu (one per key bit width, so they build in parallel).
// What the kernels compute and how is described at the top of tq_polar.cu.
#pragma once

#include <cfloat>
#include <cmath>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {


constexpr float kPolarLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1/sqrt(128)

// Grid tables of one bit width, passed by value.
struct PolarGrid {
  float t1[4];     // level 1: tan^2 of the edges inside a quadrant, index 1..m-1 (m = 2^b / 4)
  float th[16];    // levels >= 2: tan^2 of the edges k pi / 2^(b+1), index 1..2^b-1
  float cs1[32];   // level 1 midpoints: (cos, sin) of theta_hat_k, k < 2^b, interleaved
  float csh[32];   // levels >= 2: (cos, sin) of theta_hat_k
  uint8_t ucell[256];  // levels >= 2: #{k : th[k] <= i / 256}, at most one edge per cell
};

// ------------------------------------------------------------------ direction

// Code in record slot SLOT of BITS-bit codes held as 32-bit words.
template <int BITS, int SLOT>
__device__ __forceinline__ uint32_t slot_code(const uint32_t (&w)[16]) {
  constexpr int bit = BITS * SLOT, word = bit >> 5, sh = bit & 31;
  uint32_t v = w[word] >> sh;
  if constexpr (sh + BITS > 32) v |= w[word + 1] << (32 - sh);
  return v & ((1u << BITS) - 1u);
}

// Depth-first expansion of the unit direction below node NODE of level LEVEL
// (level 0 = coordinates): child 2 NODE takes val * cos(theta_hat), child
// 2 NODE + 1 takes val * sin(theta_hat).  cs1 / csh: interleaved (cos, sin)
// tables of the level-1 and the higher-level grids in shared memory.
template <int BITS, int LEVEL, int NODE, typename Leaf>
__device__ __forceinline__ void expand(const uint32_t (&w)[16], float val, const float* cs1, const float* csh,
                                       Leaf& leaf) {
  if constexpr (LEVEL == 0) {
    leaf.template at<NODE>(val);
  } else {
    constexpr int slot = kD - (kD >> (LEVEL - 1)) + NODE;
    const uint32_t code = slot_code<BITS, slot>(w);
    const float2 cs = *reinterpret_cast<const float2*>((LEVEL == 1 ? cs1 : csh) + 2 * code);
    expand<BITS, LEVEL - 1, 2 * NODE>(w, val * cs.x, cs1, csh, leaf);
    expand<BITS, LEVEL - 1, 2 * NODE + 1>(w, val * cs.y, cs1, csh, leaf);
  }
}

// The same expansion in packed fp32 pairs: every node's two children come from one
// (val, val) * (cos, sin) product; level-1 nodes hand the coordinate pair
// (y_hat_{2 NODE}, y_hat_{2 NODE + 1}) to leaf.pair<NODE>.
template <int BITS, int LEVEL, int NODE, typename Leaf>
__device__ __forceinline__ void expand2(const uint32_t (&w)[16], float val, const float* cs1, const float* csh,
                                        Leaf& leaf) {
  constexpr int slot = kD - (kD >> (LEVEL - 1)) + NODE;
  const uint32_t code = slot_code<BITS, slot>(w);
  const float2 cs = *reinterpret_cast<const float2*>((LEVEL == 1 ? cs1 : csh) + 2 * code);
  const float2 ch = __fmul2_rn(make_float2(val, val), cs);
  if constexpr (LEVEL == 1) {
    leaf.template pair<NODE>(ch);
  } else {
    expand2<BITS, LEVEL - 1, 2 * NODE>(w, ch.x, cs1, csh, leaf);
    expand2<BITS, LEVEL - 1, 2 * NODE + 1>(w, ch.y, cs1, csh, leaf);
  }
}

// ------------------------------------------------------------------ decode

constexpr int kPolarNW = 4;          // warps per decode CTA (two CTAs per SM)
constexpr int kPolarStages = 2;      // ring depth (stages of two blocks)
constexpr int kPolarPage = 16 * 64 + 32;  // a page in shared memory: 16 records padded to 64 B + radii
constexpr int kPolarStage = 4 * kPolarPage;  // K and V pages of two blocks

struct PolarDecodeArgs {
  const uint8_t* kpool;
  const uint8_t* vpool;
  int kpage, vpage;        // page bytes in the pools
  int Hkv, Hq, g, ngroups, splits;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* ctx_lens;
  const void* q;
  int q_bf16;
  float q_scale;           // sm_scale * log2(e) / sqrt(d) (the FWHT is unnormalised)
  const float* signs;
  float* part;             // [B][Hq][splits][d]
  float* ml;               // [B][Hq][splits][2]
  int64_t chunks;
  unsigned* status;
  float cs1k[32], cshk[32], cs1v[32], cshv[32];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Copies one page (16 records of 16*BITS bytes + 16 fp16 radii) into its shared
// layout: record t at t * 64, its 16-byte chunk c at position c ^ ((t >> 1) & 3)
// (conflict-free 16-byte reads of one record per lane), radii at 1024.
template <int BITS>
__device__ __forceinline__ void copy_page(uint8_t* dst, const uint8_t* src, int lane) {
  constexpr int n_rec = 16 * BITS;  // record chunks
  for (int ci = lane; ci < n_rec + 2; ci += 32) {
    if (ci < n_rec) {
      const int t = ci / BITS, c = ci - t * BITS;
      cp_async16(dst + t * 64 + ((c ^ ((t >> 1) & 3)) << 4), src + 16 * ci);
    } else {
      cp_async16(dst + 1024 + 16 * (ci - n_rec), src + 16 * ci);
    }
  }
}

template <int BITS>
__device__ __forceinline__ void load_record(const uint8_t* page, int t, uint32_t (&w)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < BITS) {
      const uint4 v = *reinterpret_cast<const uint4*>(page + t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
      w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    } else {
      w[4 * c] = w[4 * c + 1] = w[4 * c + 2] = w[4 * c + 3] = 0u;
    }
  }
}

// fp16 pair (low half = a, high half = b), each rounded to nearest.
__device__ __forceinline__ uint32_t half2_bits(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 hi/lo split of a pair: hi = fp16(v), lo = fp16(v - hi); returns hi or lo.
__device__ __forceinline__ uint32_t half2_part(float a, float b, bool lo) {
  if (!lo) return half2_bits(a, b);
  return half2_bits(a - __half2float(__float2half_rn(a)), b - __half2float(__float2half_rn(b)));
}

// Key leaf: s2[h] += (y_hat_{2i}, y_hat_{2i+1}) * (q'_{2i,h}, q'_{2i+1,h}) in packed
// fp32 pairs (queries stored [pair][NH][2]); the logit of head h is s2[h].x + s2[h].y.
template <int NH>
struct KeyLeaf {
  float2 s2[NH];
  const float* qs;
  template <int I>
  __device__ __forceinline__ void pair(float2 v) {
#pragma unroll
    for (int h2 = 0; h2 < NH / 2; ++h2) {
      const float4 qv = *reinterpret_cast<const float4*>(qs + (I * NH + 2 * h2) * 2);
      s2[2 * h2] = __ffma2_rn(v, make_float2(qv.x, qv.y), s2[2 * h2]);
      s2[2 * h2 + 1] = __ffma2_rn(v, make_float2(qv.z, qv.w), s2[2 * h2 + 1]);
    }
  }
};

// Value leaf: one half (64 coordinates) of the direction as fp16 in its token's
// row (128 B) of the [32][64] tile: 16-byte chunk c (coordinates 8c .. 8c + 7 of
// the half) at position c ^ (row & 7), so the chunk stores of a warp and the
// ldmatrix rows never share banks.
struct HalfLeaf {
  uint32_t h[4];
  uint8_t* row;
  int sw;
  template <int I>
  __device__ __forceinline__ void pair(float2 v) {
    h[I & 3] = half2_bits(v.x, v.y);
    if constexpr ((I & 3) == 3)
      *reinterpret_cast<uint4*>(row + ((((I >> 2) & 7) ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
  }
};

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&d)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One warp per chunk = (sequence b, KV head, head group, split s).  Per stage of
// two blocks (32 tokens) lane t handles token t: it rebuilds the unit direction of
// the key in fp32 pairs and dots it with the rotated queries (logits in fp32),
// then rebuilds the value direction, one half of 64 coordinates at a time, into an
// fp16 tile; acc^T (128 x 8 per n-tile) += V_hat^T x W on tensor cores with W = p r_V split into fp16 hi / lo columns
// (8 columns = 4 heads x {hi, lo}).  In the MMA layout lane (g, t) owns head
// 4 nt + t, coordinates 16 mt + g and 16 mt + g + 8.
template <int BK, int BV, int NH>
__global__ void __launch_bounds__(kPolarNW * 32, NH == 4 ? 3 : 2) k_polar_decode(PolarDecodeArgs a) {
  constexpr int NT = NH / 4;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(16) float tabs[128];  // cs1k, cshk, cs1v, cshv (static: lookups address code * 8 + constant)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < 32) {
    tabs[threadIdx.x] = a.cs1k[threadIdx.x];
    tabs[32 + threadIdx.x] = a.cshk[threadIdx.x];
    tabs[64 + threadIdx.x] = a.cs1v[threadIdx.x];
    tabs[96 + threadIdx.x] = a.cshv[threadIdx.x];
  }
  constexpr int kWarpBytes = kPolarStages * kPolarStage + (128 + 32) * NH * 4 + 32 * 128;
  uint8_t* wbase = smem_raw + warp * kWarpBytes;
  uint8_t* ring = wbase;
  float* qs = reinterpret_cast<float*>(wbase + kPolarStages * kPolarStage);  // [64 pairs][NH][2]
  float* wts = qs + 128 * NH;                                                  // [32][NH]
  uint8_t* tile = reinterpret_cast<uint8_t*>(wts + 32 * NH);                   // [32][128 B] fp16
  __syncthreads();
  const int64_t chunk = (int64_t)blockIdx.x * kPolarNW + warp;
  if (chunk >= a.chunks) return;
  const int s = (int)(chunk % a.splits);
  const int64_t unit = chunk / a.splits;
  const int hg = (int)(unit % a.ngroups);
  const int kvh = (int)((unit / a.ngroups) % a.Hkv);
  const int b = (int)(unit / ((int64_t)a.ngroups * a.Hkv));
  const int h0 = kvh * a.g + hg * NH;
  const int nh = min(NH, a.g - hg * NH);
  int ctx = __ldg(a.ctx_lens + b);
  if (ctx < 0 || ctx > a.max_blocks * 16) {
    if (lane == 0) flag_status(a.status, TQ_DEV_BAD_CONTEXT);
    ctx = 0;
  }
  const int nblk = (ctx + 15) >> 4;
  const int j0 = (int)((int64_t)s * nblk / a.splits), j1 = (int)((int64_t)(s + 1) * nblk / a.splits);

  // rotated, scaled queries: q'[j][h] = scale * (H D q_h)_j, stored by coordinate pair
  for (int h = 0; h < NH; ++h) {
    float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (h < nh) {
      const int64_t row = (int64_t)b * a.Hq + h0 + h;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * lane + k;
        const float qv = a.q_bf16 ? load_elem(reinterpret_cast<const __nv_bfloat16*>(a.q) + row * kD + j)
                                  : load_elem(reinterpret_cast<const float*>(a.q) + row * kD + j);
        y[k] = qv * __ldg(a.signs + j);
      }
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
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * lane + k;
      qs[((j >> 1) * NH + h) * 2 + (j & 1)] = y[k] * a.q_scale;
    }
  }
  __syncwarp();

  const int n_my = j1 - j0;
  const int n_st = (n_my + 1) >> 1;
  const int32_t* bt = a.block_table + (int64_t)b * a.max_blocks;
  auto block_id = [&](int jb) -> int64_t {
    if (jb >= j1) return -1;
    const int64_t id = __ldg(bt + jb);
    if (id < 0 || id >= a.num_blocks) {
      flag_status(a.status, TQ_DEV_BAD_BLOCK);
      return -1;
    }
    return id;
  };
  auto issue = [&](int st) {
    if (st < n_st) {
      uint8_t* dst = ring + (st % kPolarStages) * kPolarStage;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int64_t id = block_id(j0 + 2 * st + half);
        if (id < 0) continue;
        copy_page<BK>(dst + half * kPolarPage, a.kpool + (id * a.Hkv + kvh) * (int64_t)a.kpage, lane);
        copy_page<BV>(dst + (2 + half) * kPolarPage, a.vpool + (id * a.Hkv + kvh) * (int64_t)a.vpage, lane);
      }
    }
    cp_async_commit();
  };
  issue(0);

  float M[NH], lsum[NH], acc[8][NT][4];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    M[h] = -INFINITY;
    lsum[h] = 0.0f;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[mt][nt][k] = 0.0f;
  const float* cs1k = tabs; const float* cshk = tabs + 32;
  const float* cs1v = tabs + 64; const float* cshv = tabs + 96;
  const int half = lane >> 4, t16 = lane & 15;
  const int g = lane >> 2, tq = lane & 3;
  HalfLeaf hl;
  hl.row = tile + lane * 128;
  hl.sw = lane & 7;
  const uint32_t tile_u = (uint32_t)__cvta_generic_to_shared(tile);
  const int mat = lane >> 3, mr = lane & 7;
  // ldmatrix rows of the transposed value tiles (token 16 kt + mr + 8 (mat >> 1))
  const uint32_t v_row = tile_u + (uint32_t)((mr + ((mat >> 1) << 3)) * 128);

  for (int st = 0; st < n_st; ++st) {
    issue(st + 1);
    cp_async_wait<1>();
    __syncwarp();
    const uint8_t* sbuf = ring + (st % kPolarStages) * kPolarStage;
    const int jb = j0 + 2 * st + half;
    bool valid = jb < j1 && jb * 16 + t16 < ctx;
    if (valid) {  // the block id was checked when its pages were requested
      const int64_t id = __ldg(bt + jb);
      valid = id >= 0 && id < a.num_blocks;
    }
    // keys: fp32 logits in log2 units
    const uint8_t* kp = sbuf + half * kPolarPage;
    uint32_t w[16];
    load_record<BK>(kp, t16, w);
    const float rk = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(kp + 1024 + 2 * t16)));
    KeyLeaf<NH> kl;
    kl.qs = qs;
#pragma unroll
    for (int h = 0; h < NH; ++h) kl.s2[h] = make_float2(0.0f, 0.0f);
    expand2<BK, 7, 0>(w, 1.0f, cs1k, cshk, kl);
    const uint8_t* vp = sbuf + (2 + half) * kPolarPage;
    const float rv = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(vp + 1024 + 2 * t16)));
    float corr[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float sc = valid ? (kl.s2[h].x + kl.s2[h].y) * rk : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(M[h], mx);
      corr[h] = (M[h] == -INFINITY) ? 0.0f : ex2(M[h] - mn);
      const float p = valid ? ex2(sc - mn) : 0.0f;
      lsum[h] = lsum[h] * corr[h] + p;
      M[h] = mn;
      wts[lane * NH + h] = valid ? p * rv : 0.0f;
    }
    bool moved = false;  // warp-uniform: the running maxima are
#pragma unroll
    for (int h = 0; h < NH; ++h) moved |= corr[h] != 1.0f;
    if (moved) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float c = tq == 0 ? corr[4 * nt] : tq == 1 ? corr[4 * nt + 1] : tq == 2 ? corr[4 * nt + 2] : corr[4 * nt + 3];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[mt][nt][k] *= c;
      }
    }
    // values: directions to the fp16 tile one half at a time, then acc^T += V_hat^T W
    load_record<BV>(vp, t16, w);
    __syncwarp();  // weights of every token written
    uint32_t bp[2][NT][2];
#pragma unroll
    for (int kt = 0; kt < 2; ++kt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hd = 4 * nt + (g >> 1), t0 = 16 * kt + 2 * tq;
        bp[kt][nt][0] = half2_part(wts[t0 * NH + hd], wts[(t0 + 1) * NH + hd], g & 1);
        bp[kt][nt][1] = half2_part(wts[(t0 + 8) * NH + hd], wts[(t0 + 9) * NH + hd], g & 1);
      }
    const float2 cs7 = *reinterpret_cast<const float2*>(cshv + 2 * slot_code<BV, kD - 2>(w));
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      if (hv == 0) expand2<BV, 6, 0>(w, cs7.x, cs1v, cshv, hl);
      else expand2<BV, 6, 1>(w, cs7.y, cs1v, cshv, hl);
      __syncwarp();
#pragma unroll
      for (int kt = 0; kt < 2; ++kt)
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          uint32_t af[4];
          const int c = 2 * m4 + (mat & 1);
          ldsm_x4_t(v_row + (uint32_t)(kt * 16 * 128) + (uint32_t)((c ^ mr) << 4), af);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16(acc[4 * hv + m4][nt], af, bp[kt][nt][0], bp[kt][nt][1]);
        }
      __syncwarp();
    }
  }
  cp_async_wait<0>();

  // partials: unnormalised acc of head 4 nt + tq (hi + lo columns), (max, denominator)
#pragma unroll
  for (int h = 0; h < NH; ++h) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], o);
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + tq;
    if (h < nh) {
      const int64_t slot = ((int64_t)b * a.Hq + h0 + h) * a.splits + s;
      float* pr = a.part + slot * kD;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        pr[16 * mt + g] = acc[mt][nt][0] + acc[mt][nt][1];
        pr[16 * mt + g + 8] = acc[mt][nt][2] + acc[mt][nt][3];
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (h < nh) {
        const int64_t slot = ((int64_t)b * a.Hq + h0 + h) * a.splits + s;
        a.ml[2 * slot] = M[h];
        a.ml[2 * slot + 1] = lsum[h];
      }
    }
  }
}

template <int BK, int BV, int NH>
cudaError_t run_polar_decode(const PolarDecodeArgs& a, cudaStream_t st) {
  auto kern = k_polar_decode<BK, BV, NH>;
  constexpr int kWarpBytes = kPolarStages * kPolarStage + (128 + 32) * NH * 4 + 32 * 128;
  constexpr size_t smem = (size_t)kPolarNW * kWarpBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = (a.chunks + kPolarNW - 1) / kPolarNW;
  kern<<<(unsigned)grid, kPolarNW * 32, smem, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

// Decode launch of one key bit width (one translation unit per BK keeps the
// build parallel): the value width and the heads per warp are dispatched here.
template <int BK>
cudaError_t polar_decode_bk(const PolarDecodeArgs& a, int bv, int nh, cudaStream_t st) {
  if (nh == 4) {
    switch (bv) {
      case 2: return run_polar_decode<BK, 2, 4>(a, st);
      case 3: return run_polar_decode<BK, 3, 4>(a, st);
      default: return run_polar_decode<BK, 4, 4>(a, st);
    }
  }
  switch (bv) {
    case 2: return run_polar_decode<BK, 2, 8>(a, st);
    case 3: return run_polar_decode<BK, 3, 8>(a, st);
    default: return run_polar_decode<BK, 4, 8>(a, st);
  }
}
extern template cudaError_t polar_decode_bk<2>(const PolarDecodeArgs&, int, int, cudaStream_t);
extern template cudaError_t polar_decode_bk<3>(const PolarDecodeArgs&, int, int, cudaStream_t);
extern template cudaError_t polar_decode_bk<4>(const PolarDecodeArgs&, int, int, cudaStream_t);

}  // namespace tq
