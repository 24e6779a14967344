/*
 * tq.h -- C ABI of libtq: TurboQuant quantized KV cache on NVIDIA GB300 (sm_103a).
 *
 * This header is the written specification both the CUDA library and the
 * independent CPU oracle are built from.  Sources are cited by page title and
 * section:
 *   [P1] issoh.co.jp "TurboQuantとは？vLLM・Ollama・LM Studioの対応状況と使い方"
 *   [P2] ai-navigate-news.com, the turboquant-vllm article
 *   [P3] lilting.ch "HypuraのNVMeストリーミングとTurboQuantのKVキャッシュ量子化"
 *   [P4] qiita.com, AMD's mixed BF16/4-bit KV cache in LMCache
 *
 * ------------------------------------------------------------------------
 * Method (what the library computes)
 *
 *  Stage 1 ([P1] §第1段, §第2段 "_nc"): every key/value vector x in R^d is
 *  rotated by a per-layer random rotation Pi, divided by its norm, and each
 *  coordinate is replaced by the index of its Lloyd-Max cell; the fp32 norm
 *  correction gamma is stored beside the codes ([P2] "Bugs Nobody Else Has
 *  Found": fp32, not fp16):
 *      n = ||x||,  y = Pi x / n,  idx_j = #{ i : y_j >= beta_i },
 *      gamma = n / ||c[idx]||   (TQ_NORM_CORRECTED)   or  n  (TQ_NORM_RAW),
 *      x_hat = gamma Pi^T c[idx];   zero vector: gamma = 0, idx_j = 2^(b-1).
 *  Ties (y_j == beta_i) go to the upper cell.
 *
 *  Stage 2, optional for keys ([P3] "QJL: Johnson-Lindenstrauss変換で残差を
 *  1ビット補正する"): r = Pi x - gamma c[idx] (rotated domain), store the
 *  m = d sign bits sigma_i = [(S r)_i >= 0] and rho = ||r|| (fp32); S is an
 *  m x d matrix of iid N(0,1) shared by all layers and heads.  Score estimate:
 *      <q, x> ~= gamma <Pi q, c[idx]> + sqrt(pi/2)/m rho sum_i (2 sigma_i - 1)(S Pi q)_i.
 *
 *  Decode attention on the packed cache (no dequantized K/V written to HBM):
 *      q' = Pi q once per query head; s_t = sm_scale * gamma_t <q', c_K[idx_t]>
 *      (+ the QJL term); online softmax over the context; the value sum is
 *      accumulated in the rotated domain, sum_t p_t gamma'_t c_V[idx'_t];
 *      one inverse rotation Pi^T per query head at the end.
 *  Query head h reads KV head h / (H_q / H_kv) (grouped-query attention).
 *  bf16 layers ([P1] §起動コマンド: the first and last two layers of dense
 *  models stay at full precision; [P4] layout table, 512 B per token and head)
 *  hold raw bf16 K/V and are attended without rotation.
 *  k8v4 layers ([P1] §プリセット: FP8 keys with 4-bit TurboQuant values, the
 *  error of the method coming almost entirely from the keys) store each key
 *  coordinate as FP8 E4M3 (no rotation, no scale) and the values as above;
 *  decode scores s_t = sm_scale <q, fp8(k_t)> with the raw query and keeps the
 *  rotated-domain value sum and the one inverse rotation per query head.
 *  Polar layers ([P3] "PolarQuant: 極座標変換で量子化定数を不要にする"): the
 *  vector is rotated (Hadamard Pi), then turned into polar coordinates
 *  recursively -- coordinate pairs give d/2 radii and d/2 angles, the radii
 *  are paired again, ... -- until one radius and d - 1 angles remain; every
 *  angle is quantized on one fixed uniform grid (no per-block constants) and
 *  the radius is kept as fp16 (2 bytes per vector):
 *      y = Pi x;  level 1: theta_{1,i} = atan2(y_{2i+1}, y_{2i}), i < d/2,
 *      rho_{1,i} = |(y_{2i}, y_{2i+1})|;  level l >= 2:
 *      theta_{l,i} = atan2(rho_{l-1,2i+1}, rho_{l-1,2i}) in [0, pi/2];
 *      r = fp16(||x||) (round to nearest even).
 *    Codes (b bits per angle): level 1 on the whole circle,
 *      k = floor(phi / (2 pi / 2^b)), phi = theta + pi taken mod 2 pi in
 *      [0, 2 pi) (theta = pi and theta = -pi give k = 0);
 *    levels >= 2 on [0, pi/2]: k = min(floor(theta / (pi / 2^(b+1))), 2^b - 1).
 *    A pair whose two entries are both zero has theta = 0.  Reconstruction
 *    takes every angle at its cell's midpoint; coordinate j of the unit
 *    direction is the product over levels l = 1..log2 d of cos(theta_hat) if
 *    bit l-1 of j is 0, sin(theta_hat) if it is 1, for the level-l angle
 *    number j >> l; x_hat = r Pi^T y_hat (||x_hat|| = r).  Decode scores are
 *    s_t = sm_scale r_t <Pi q, y_hat_t>; values are summed in the rotated
 *    domain as for the packed layers.
 *
 * ------------------------------------------------------------------------
 * Readings of the pages (they leave these open; the library and the oracle
 * both follow them)
 *
 *  Random streams: SplitMix64 (Vigna).  state0 = seed ^ ((kind<<32) + layer)
 *    * 0x9E3779B97F4A7C15 (mod 2^64); next: state += 0x9E3779B97F4A7C15,
 *    z = state, z = (z^(z>>30))*0xBF58476D1CE4E5B9, z = (z^(z>>27))*
 *    0x94D049BB133111EB, out = z^(z>>31).  Sign i = -1 iff bit 63 of draw i.
 *    Uniform = (draw>>11) * 2^-53.  Gaussians: Box-Muller on consecutive
 *    uniform pairs (u1, u2): r = sqrt(-2 ln(1-u1)), g0 = r cos(2 pi u2),
 *    g1 = r sin(2 pi u2), filling matrices row-major.
 *  Hadamard rotation (kind 1): Pi = H_d diag(s) / sqrt(d), H_d Sylvester.
 *  Dense rotation (kind 2): G = d x d Gaussians; Pi = Q diag(sign(diag R))
 *    for G = Q R (the unique Haar Q).
 *  QJL projection (kind 3, layer 0): S = d x d Gaussians (m = d).
 *  Codebook: Lloyd-Max for the density of one coordinate of a uniform unit
 *    vector in R^d, f(t) ~ (1 - t^2)^((d-3)/2); Lloyd iteration in fp64 to
 *    max |delta c| < 1e-15; centroids emitted in fp32 with the upper half
 *    mirrored (c[2^b-1-i] = -c[i] exactly); boundaries
 *    beta_i = fp32(fp32(c_i + c_{i+1}) * 0.5).
 *  FP8 keys (k8v4): E4M3 -- sign, 4 exponent bits with bias 7, 3 mantissa
 *    bits, subnormals m 2^-9, no infinities, S.1111.111 = NaN, largest finite
 *    448; encoding rounds to nearest, ties to even, and saturates finite
 *    overflow and infinities to +-448 (NaN stays NaN).
 *  Packing: LSB-first bitstream; code j in bits [b j, b j + b) of the record,
 *    bit k of a record = bit (k mod 8) of byte (k div 8).  For b = 4 this is
 *    the 'codes[i] | codes[i+1] << 4' of [P4]'s worked example.
 *
 * ------------------------------------------------------------------------
 * Memory layout (device, owned by the caller)
 *
 *  Block size 16 tokens.  slot = block * 16 + offset (vLLM-style slot mapping;
 *  slot < 0 means "skip this token").
 *  Packed pool:  [num_blocks][num_kv_heads][page_bytes]; one page per
 *  (block, kv head):
 *      [16 records of d*b/8 code bytes][16 x fp32 gamma]
 *      keys with QJL add: [16 x d/8 sign bytes][16 x fp32 rho]
 *    d = 128: 1088 B (4-bit), 832 B (3-bit), 576 B (2-bit), 896 B (2-bit+QJL).
 *  bf16 pool: [num_blocks][num_kv_heads][16][d] bf16 (4096 B per page).
 *  k8v4 key pool: [num_blocks][num_kv_heads][16][d] FP8 E4M3 bytes (2048 B
 *  per page, nothing else); its value pool is a packed pool of bits_v.
 *  Polar pools (keys with bits_k, values with bits_v): one page per (block,
 *  kv head) = [16 records of d*b/8 bytes][16 x fp16 radius]; record slot s
 *  holds angle code s in the packed bitstream above, slots ordered by level
 *  (level 1 angles 0..d/2-1, then level 2, ..., the last level's one angle at
 *  slot d-2) and slot d-1 = 0.  d = 128: 1056 B (4-bit), 800 B (3-bit),
 *  544 B (2-bit).
 *  Pools must be 16-byte aligned.
 *
 * ------------------------------------------------------------------------
 * Conventions for every call
 *
 *  - Device pointers are raw CUDA device addresses; host pointers are marked.
 *  - Calls that take a stream enqueue asynchronously on it (a cudaStream_t
 *    passed as void*; NULL = legacy default stream) and never synchronize,
 *    except tq_get_device_status.
 *  - The library never allocates device memory (scratch is the caller's
 *    workspace) and keeps no pointer past the call.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing and returns a status != TQ_OK; tq_last_error() then
 *    returns a message (thread-local, valid until the next call).
 *  - Values that live on the device (slot mappings, block tables, context
 *    lengths) are range-checked inside the kernels: an out-of-range entry is
 *    skipped and recorded in a sticky per-device status word read by
 *    tq_get_device_status.  Kernels never trap.
 *  - Only head_dim = 128 and block_size = 16 are implemented.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_FORMAT_VERSION 1u
#define TQ_BLOCK_SIZE 16
#define TQ_HEAD_DIM 128
#define TQ_MAX_GROUP 8 /* query heads one decode warp handles; larger GQA groups are split into groups of 8 */

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,  /* bad argument; nothing launched */
  TQ_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim != 128) */
  TQ_ERR_WORKSPACE = 3,    /* workspace missing or too small */
  TQ_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  TQ_ERR_DEVICE = 5,       /* the device status word reported a problem */
  TQ_ERR_VERSION = 6       /* descriptor format_version mismatch */
} tq_status;

/* element types of q / k / v / out */
enum { TQ_F32 = 0, TQ_BF16 = 1 };

/* rotation / random stream kinds */
enum { TQ_ROT_HADAMARD = 1, TQ_ROT_DENSE = 2, TQ_RNG_QJL = 3 };

/* layer storage */
enum { TQ_KV_PACKED = 0, TQ_KV_BF16 = 1, TQ_KV_K8V4 = 2, TQ_KV_POLAR = 3 };

/* norm handling */
enum { TQ_NORM_CORRECTED = 0, TQ_NORM_RAW = 1 };

/* device status codes (bit flags, sticky until read) */
enum {
  TQ_DEV_BAD_SLOT = 1,        /* slot >= num_blocks * 16 in an append/dequantize */
  TQ_DEV_BAD_BLOCK = 2,       /* block table entry outside [0, num_blocks) */
  TQ_DEV_BAD_CONTEXT = 4,     /* context length < 0 or > max_blocks_per_seq * 16 */
  TQ_DEV_WAIT_TIMEOUT = 8,    /* a bounded wait on a copy gave up */
  TQ_DEV_LAYOUT = 16          /* decode found less shared memory than its layout needs (no work done) */
};

typedef struct {
  int32_t kv_format; /* TQ_KV_PACKED, TQ_KV_BF16, TQ_KV_K8V4 or TQ_KV_POLAR */
  int32_t bits_k;    /* packed: 2, 3 or 4; k8v4: 8 (FP8 E4M3 keys); polar: 2, 3 or 4 bits per angle */
  int32_t bits_v;    /* packed, k8v4 and polar: 2, 3 or 4 */
  int32_t qjl_k;     /* packed: 1 = keys carry the 1-bit QJL residual (m = head_dim); k8v4, polar: 0 */
  int32_t rot_kind;  /* packed and k8v4 (values): TQ_ROT_HADAMARD or TQ_ROT_DENSE; polar: TQ_ROT_HADAMARD */
  int32_t norm_mode; /* TQ_NORM_CORRECTED or TQ_NORM_RAW */
} tq_layer_format;

/* One descriptor per layer.  Codebooks travel by value; the tables must be
 * strictly increasing and antisymmetric (c[2^b-1-i] = -c[i], beta middle = 0),
 * as tq_make_codebook emits them.  Entries past 2^b (2^b - 1) are ignored.
 * Polar and bf16 layers ignore the codebook fields (polar angle grids are
 * fixed by the bit widths). */
typedef struct {
  uint32_t format_version; /* TQ_FORMAT_VERSION */
  int32_t head_dim;        /* 128 */
  int32_t num_kv_heads;    /* >= 1 */
  int32_t block_size;      /* 16 */
  int64_t num_blocks;      /* pages per pool */
  tq_layer_format fmt;
  void* k_cache;           /* device pool of keys (layout above) */
  void* v_cache;           /* device pool of values */
  const float* rotation;   /* device: Hadamard -> signs[d] (+1.0f / -1.0f);
                              dense -> Pi[d][d] row-major (y = Pi x); unused for bf16 */
  const float* qjl_proj;   /* device: S[d][d] row-major; required iff fmt.qjl_k */
  float centroids_k[16];
  float boundaries_k[15];
  float centroids_v[16];
  float boundaries_v[15];
} tq_cache_desc;

/* ---- set-up (host only, no GPU needed) ---------------------------------- */

/* Lloyd-Max codebook for one coordinate of a rotated unit vector in R^head_dim
 * ([P1] §第1段; density and emission rule above).  Host outputs:
 * centroids[2^bits], boundaries[2^bits - 1].  bits in 1..4. */
tq_status tq_make_codebook(int head_dim, int bits, float* centroids, float* boundaries);

/* Seeded matrices ([P1] §第1段, §llama.cpp本家; [P3] QJL section).  Host output:
 *   TQ_ROT_HADAMARD: out[head_dim] = signs s (+-1.0f); Pi = H diag(s)/sqrt(d)
 *   TQ_ROT_DENSE:    out[head_dim*head_dim] = Pi row-major (Haar, see above)
 *   TQ_RNG_QJL:      out[head_dim*head_dim] = S row-major (layer ignored: 0)
 * head_dim must be a power of two (Hadamard) or 1..1024 (dense, QJL). */
tq_status tq_make_rotation(int kind, int head_dim, uint64_t seed, int layer, float* out);

/* Bytes of one page (one block of one KV head) of the K (which = 0) or V
 * (which = 1) pool; 0 if the descriptor is invalid. */
size_t tq_page_bytes(const tq_cache_desc* desc, int which);

/* ---- hot path ----------------------------------------------------------- */

/* Quantize-on-append ([P1] §第1段/§第2段; [P3] online per-token quantization):
 * k, v: device [n_tokens][num_kv_heads][head_dim] of in_dtype (TQ_F32 or
 * TQ_BF16); either may be NULL to append only the other.  slot_mapping:
 * device int64[n_tokens]; token t goes to slot_mapping[t] (skipped if < 0).
 * Packed layers store codes + gamma (+ QJL for keys); bf16 layers store the
 * values rounded to bf16.  Writes only the records of the given slots. */
tq_status tq_quantize_append(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                             const int64_t* slot_mapping, int64_t n_tokens, void* stream);

/* Quantize-on-append of the same tokens into several layers at once (a batched
 * prefill): descs: host array of n_layers descriptors of distinct caches; k, v:
 * host arrays of n_layers device pointers, [n_tokens][num_kv_heads][head_dim]
 * of in_dtype per layer (either array may be NULL to append only the other);
 * slot_mapping, n_tokens: as tq_quantize_append, shared by all layers.  The
 * result equals n_layers tq_quantize_append calls in order.  Every layer is
 * checked before anything is launched.  Since the layers share no memory that
 * the appends write, each layer's kernel after the first is launched as a
 * programmatic dependent of the previous one and may start while it finishes;
 * the inputs must therefore be ready when the call is enqueued (written by work
 * that precedes the call on the stream), as for any kernel. */
tq_status tq_quantize_append_layers(const tq_cache_desc* const* descs, int n_layers, const void* const* k,
                                    const void* const* v, int in_dtype, const int64_t* slot_mapping,
                                    int64_t n_tokens, void* stream);

/* The quantizer alone, fed rotated unit coordinates: y: device fp32
 * [n_tokens][num_kv_heads][head_dim] (y = Pi x / ||x||), norms: device fp32
 * [n_tokens][num_kv_heads] (||x||).  Writes codes and gamma of the K
 * (which = 0) or V (which = 1) pool exactly as tq_quantize_append would from
 * the same y (no QJL residual).  Packed layers only.  It runs the quantizer of
 * the kernel a bf16 append of the same layer and size would run (the cell-table
 * quantizer of the bulk kernels for dense layers and for Hadamard calls of at
 * least 24,576 vectors, the boundary search of the per-quad kernel otherwise),
 * so every append quantizer can be checked on exact inputs; all of them give
 * the same codes for the same y. */
tq_status tq_quantize_rotated(const tq_cache_desc* desc, int which, const float* y, const float* norms,
                              const int64_t* slot_mapping, int64_t n_tokens, void* stream);

/* Number of context splits decode uses when num_splits == 0 (depends on the
 * current device's SM count); 0 on error. */
int tq_auto_splits(const tq_cache_desc* desc, int batch, int num_q_heads, int max_blocks_per_seq);

/* Workspace bytes tq_decode_attention needs for these sizes (num_splits = 0:
 * the automatic choice above).  0 on error.  The first 64 KiB of every
 * workspace (more only for shapes with over 16384 (sequence, query head)
 * rows) hold per-(sequence, KV head) chunk counters at a fixed place. */
size_t tq_workspace_bytes(const tq_cache_desc* desc, int batch, int num_q_heads, int max_blocks_per_seq,
                          int num_splits);

/* Decode attention over the cache (see "Method"):
 * q: device [batch][num_q_heads][head_dim] (q_dtype TQ_F32 / TQ_BF16);
 * block_table: device int32 [batch][max_blocks_per_seq]; context_lens: device
 * int32 [batch] (0 gives a zero output row); out: device
 * [batch][num_q_heads][head_dim] (out_dtype); workspace: device scratch of at
 * least tq_workspace_bytes(...) bytes, 256-byte aligned, all zero before the
 * first call that uses it (e.g. cudaMemsetAsync once after allocating it).
 * Every call leaves the counter region at zero again, so one workspace serves
 * any sequence of calls, shapes and layers without clearing; memory that held
 * anything else in between must be zero-filled again.  num_q_heads must be a
 * multiple of num_kv_heads (any group size: a group above TQ_MAX_GROUP heads
 * is split into warps of 8 heads that each stream the KV head's pages).
 * num_splits: 0 = automatic, else the
 * number of contiguous ranges each (sequence, KV head) is split into;
 * results agree for every split count up to fp32 rounding.  The ranges cut the
 * block-table row (max_blocks_per_seq entries), so a sequence's block ids are
 * read while its context length is still in flight; a row more than a third
 * wider than the sequence's context (a table padded to a maximum length) is
 * cut over the context instead, at the cost of reading the block ids after it.
 * Either way the output is the same function of the inputs. */
tq_status tq_decode_attention(const tq_cache_desc* desc, const void* q, int q_dtype, int batch,
                              int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* context_lens, float sm_scale, void* out, int out_dtype,
                              void* workspace, size_t workspace_bytes, int num_splits, void* stream);

/* One decode step of a layer: tq_quantize_append(desc, k, v, in_dtype,
 * slot_mapping, n_tokens) followed by tq_decode_attention(desc, q, ...) on the
 * same stream, with the same arguments, results and errors as those two calls
 * made in that order (every argument of both is checked before anything is
 * launched).  The decode kernel is launched as a programmatic dependent of the
 * append: its prologue (context lengths, block ids, query rotation, code
 * tables) runs while the append is still writing, and it waits for the append
 * to finish before it reads any page.  For dense-rotation and QJL layers the
 * query pass (q' = Pi q, S q') is the append's dependent instead and the decode
 * that pass's; the pass reads only q and writes only the workspace, and it
 * completes only after the append.  q, block_table and context_lens are
 * therefore read while the append runs; the append never writes them. */
tq_status tq_append_decode(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                           const int64_t* slot_mapping, int64_t n_tokens, const void* q, int q_dtype, int batch,
                           int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* context_lens, float sm_scale, void* out, int out_dtype, void* workspace,
                           size_t workspace_bytes, int num_splits, void* stream);

/* One decode step of a layer in a single kernel: the new token of every sequence
 * is quantized by the decode kernel itself and attended to in the same call.
 * k_new, v_new: device [batch][num_kv_heads][head_dim] (in_dtype TQ_F32 or
 * TQ_BF16, 16-byte aligned); context_lens[b] already counts the new token, which
 * is written at position context_lens[b] - 1 of sequence b (slot block_table[b]
 * [(context_lens[b] - 1) / 16] * 16 + (context_lens[b] - 1) % 16); a sequence
 * with context_lens[b] == 0 gets no token and a zero output row.  The record is
 * the same quantization as tq_quantize_append's ("Method"), computed by one warp
 * per (sequence, KV head) in fp32 with its own order of operations, so a code may
 * differ from the append kernels' only where y lies within the 1e-5 tie band of a
 * boundary (the same bound the append kernels meet against the exact method).
 * The warp that reads the new token's block writes the record to the cache and
 * into its own shared-memory copy of the block, so no other kernel runs and no
 * CTA waits for another.  Other arguments, the workspace contract and errors as
 * for tq_decode_attention.  Packed layers with a Hadamard rotation and without
 * QJL keys only (TQ_ERR_UNSUPPORTED otherwise); every context length must be >= 1
 * for a sequence whose token is to be appended. */
tq_status tq_decode_step(const tq_cache_desc* desc, const void* k_new, const void* v_new, int in_dtype,
                         const void* q, int q_dtype, int batch, int num_q_heads, const int32_t* block_table,
                         int max_blocks_per_seq, const int32_t* context_lens, float sm_scale, void* out,
                         int out_dtype, void* workspace, size_t workspace_bytes, int num_splits, void* stream);

/* Dequantize records ([P2] "Incremental dequantization"): slots: device int64[n];
 * out: device [n][num_kv_heads][head_dim] (out_dtype) with
 * x_hat = gamma Pi^T c[idx] of the K (which = 0) or V (which = 1) pool
 * (bf16 layers: the stored values).  Negative slots give zero rows. */
tq_status tq_dequantize(const tq_cache_desc* desc, int which, const int64_t* slots, int64_t n, void* out,
                        int out_dtype, void* stream);

/* ---- offload / restore ([P4]: LMCache copies BF16 and packed groups
 * uninterpreted, restoring exactly what was stored, T(Q(X)) = Q(X), and the
 * reader must know the format id and version of what it reads) -------------
 *
 * Image of n blocks of one layer (host memory, little-endian):
 *   bytes 0..7 "TQKVIMG1"; 8..11 TQ_FORMAT_VERSION (uint32); 12..35 the layer
 *   format (kv_format, bits_k, bits_v, qjl_k, rot_kind, norm_mode, int32);
 *   36..47 head_dim, num_kv_heads, block_size (int32); 48..55 n (int64);
 *   56..63 FNV-1a 64 of centroids_k[16], boundaries_k[15], centroids_v[16],
 *   boundaries_v[15] as fp32 bytes; then the K pages of every KV head of the
 *   listed blocks in the order listed, then their V pages in the same order.
 * The rotation (and QJL projection) of the layer are not in the image: restore
 * into a layer built with the same ones. */

/* Bytes of the image of n_blocks blocks of this layer; 0 if invalid. */
size_t tq_image_bytes(const tq_cache_desc* desc, int64_t n_blocks);

/* Copies the pages of blocks[0..n) (host int32 array, each in [0, num_blocks))
 * of both pools into image after writing its header (by the host, before this
 * call returns).  image: pinned (or managed) host memory, 16-byte aligned: the
 * pages are copied by a kernel through the image's device address.
 * image_bytes must be at least tq_image_bytes(desc, n).  Enqueued on the
 * stream; the image is complete once the stream has reached this point. */
tq_status tq_offload_blocks(const tq_cache_desc* desc, const int32_t* blocks, int64_t n, void* image,
                            size_t image_bytes, void* stream);

/* Checks the image header against the descriptor (magic, version, layer format,
 * head_dim, num_kv_heads, block_size, n, codebook hash: TQ_ERR_VERSION for a
 * version mismatch, TQ_ERR_INVALID_ARG for any other) and copies its pages into
 * blocks[0..n) (host int32 array; the same or other blocks than were offloaded).
 * image: pinned (or managed) host memory as for tq_offload_blocks.  Writes
 * nothing else of the pools.  The image must stay valid until the stream has
 * reached this point. */
tq_status tq_restore_blocks(const tq_cache_desc* desc, const int32_t* blocks, int64_t n, const void* image,
                            size_t image_bytes, void* stream);

/* Bytes of the scratch array tq_decode_attention_static keeps on every device
 * that loads the library (held until the process exits). */
#define TQ_STATIC_SCRATCH_BYTES (8u << 20)

/* Decode attention for callers that cannot allocate device memory.  The pages
 * have no counterpart for this call: it exists for code that is handed only
 * its inputs and outputs (a plugin or FFI caller inside a host application
 * that owns the device-memory budget, or a serving loop that must not call
 * cudaMalloc/cudaFree after start-up), so it cannot pass the workspace
 * tq_decode_attention needs.
 * Same arguments, result and errors as tq_decode_attention without the
 * workspace pair; the scratch is a library-owned device array of
 * TQ_STATIC_SCRATCH_BYTES.  Sizes whose scratch would exceed it are rejected
 * with TQ_ERR_WORKSPACE before anything is launched.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, that
 * device current): make it before any stream capture.  Allocates nothing.
 * All calls on a device share the array; calls that overlap on the GPU (other
 * streams, other host threads) race on it.  The array's counter region starts
 * at zero (the array is zero-filled when the library loads) and every call
 * leaves it at zero: the decode kernels contain no wait that can give up, and a
 * call that flags TQ_DEV_BAD_BLOCK or TQ_DEV_BAD_CONTEXT still completes every
 * (sequence, KV head) unit, so one faulty call does not disturb later ones. */
tq_status tq_decode_attention_static(const tq_cache_desc* desc, const void* q, int q_dtype, int batch,
                                     int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* context_lens, float sm_scale, void* out, int out_dtype,
                                     int num_splits, void* stream);

/* ---- status ------------------------------------------------------------- */

/* Synchronizes the stream, returns the sticky device status bits of the
 * current device in *code (host pointer) and clears them. */
tq_status tq_get_device_status(void* stream, int32_t* code);

/* Message describing the last failed call on this thread ("" if none). */
const char* tq_last_error(void);

/* TQ_FORMAT_VERSION of this build. */
uint32_t tq_format_version(void);

/* Number of kernels this library has enqueued in this process, all threads
 * and devices together (a host-side count taken at each launch; a launch made
 * during stream capture counts once, however often the graph is replayed). */
uint64_t tq_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
