// Offload / restore of cache blocks to host images: the stored bytes of each
// page copied uninterpreted (a copy kernel that reads or writes the pinned image
// through its device address, block ids in the kernel parameters), under a
// header that names the format, so that a restore gives back exactly what was
// stored.  The image layout and every error are specified in include/tq.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr size_t kHeaderBytes = 64;
constexpr char kMagic[8] = {'T', 'Q', 'K', 'V', 'I', 'M', 'G', '1'};

// FNV-1a, 64-bit (Fowler, Noll, Vo).
uint64_t fnv1a64(const unsigned char* p, size_t n, uint64_t h = 0xCBF29CE484222325ull) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001B3ull;
  }
  return h;
}

uint64_t codebook_hash(const tq_cache_desc& d) {
  uint64_t h = fnv1a64(reinterpret_cast<const unsigned char*>(d.centroids_k), sizeof(d.centroids_k));
  h = fnv1a64(reinterpret_cast<const unsigned char*>(d.boundaries_k), sizeof(d.boundaries_k), h);
  h = fnv1a64(reinterpret_cast<const unsigned char*>(d.centroids_v), sizeof(d.centroids_v), h);
  return fnv1a64(reinterpret_cast<const unsigned char*>(d.boundaries_v), sizeof(d.boundaries_v), h);
}

void put32(unsigned char* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
void put64(unsigned char* p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
uint32_t get32(const unsigned char* p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
  return v;
}
uint64_t get64(const unsigned char* p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
  return v;
}

void make_header(const tq_cache_desc& d, int64_t n, unsigned char* h) {
  std::memset(h, 0, kHeaderBytes);
  std::memcpy(h, kMagic, 8);
  put32(h + 8, TQ_FORMAT_VERSION);
  const int32_t f[6] = {d.fmt.kv_format, d.fmt.bits_k, d.fmt.bits_v, d.fmt.qjl_k, d.fmt.rot_kind, d.fmt.norm_mode};
  for (int i = 0; i < 6; ++i) put32(h + 12 + 4 * i, (uint32_t)f[i]);
  put32(h + 36, (uint32_t)d.head_dim);
  put32(h + 40, (uint32_t)d.num_kv_heads);
  put32(h + 44, (uint32_t)d.block_size);
  put64(h + 48, (uint64_t)n);
  put64(h + 56, codebook_hash(d));
}

tq_status check_blocks(const tq_cache_desc& d, const int32_t* blocks, int64_t n, const char* fn) {
  if (n < 0) return fail(TQ_ERR_INVALID_ARG, "%s: n < 0", fn);
  if (n > 0 && !blocks) return fail(TQ_ERR_INVALID_ARG, "%s: null blocks", fn);
  for (int64_t i = 0; i < n; ++i)
    if (blocks[i] < 0 || (int64_t)blocks[i] >= d.num_blocks)
      return fail(TQ_ERR_INVALID_ARG, "%s: blocks[%lld] = %d outside [0, %lld)", fn, (long long)i, blocks[i],
                  (long long)d.num_blocks);
  return TQ_OK;
}

// Block ids travel in the kernel parameters, kMaxIds per launch.
constexpr int kMaxIds = 1024;
struct BlockIds {
  int32_t id[kMaxIds];
};

// Copies n whole blocks (bytes_per_block each, a multiple of 16) between a pool and
// consecutive slots of an image: pool block ids.id[i] <-> image slot i.
__global__ void __launch_bounds__(256) k_copy_blocks(unsigned char* pool, unsigned char* img, BlockIds ids, int n,
                                                     size_t bytes_per_block, int to_image) {
  const size_t words = bytes_per_block / 16;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    uint4* p = reinterpret_cast<uint4*>(pool + (size_t)ids.id[i] * bytes_per_block);
    uint4* m = reinterpret_cast<uint4*>(img + (size_t)i * bytes_per_block);
    if (to_image)
      for (size_t w = threadIdx.x; w < words; w += blockDim.x) m[w] = p[w];
    else
      for (size_t w = threadIdx.x; w < words; w += blockDim.x) p[w] = m[w];
  }
}

// The image must be host memory the device can address directly (pinned or managed).
tq_status check_image_memory(const void* image, const char* fn) {
  if (reinterpret_cast<uintptr_t>(image) & 15) return fail(TQ_ERR_INVALID_ARG, "%s: image must be 16-byte aligned", fn);
  cudaPointerAttributes at;
  const cudaError_t e = cudaPointerGetAttributes(&at, image);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(TQ_ERR_INVALID_ARG, "%s: image is not memory the device can address (%s)", fn, cudaGetErrorString(e));
  }
  // the host writes / reads the header, the device the pages: pinned or managed memory
  if (at.type != cudaMemoryTypeHost && at.type != cudaMemoryTypeManaged)
    return fail(TQ_ERR_INVALID_ARG, "%s: image must be pinned (or managed) host memory", fn);
  return TQ_OK;
}

// Both pools of the listed blocks <-> the image body (K section, then V section).
tq_status copy_blocks(const tq_cache_desc& d, const int32_t* blocks, int64_t n, const void* image_body, bool to_image,
                      int num_sms, cudaStream_t st) {
  const size_t bk = (size_t)d.num_kv_heads * page_bytes_of(d, 0);  // K bytes per block
  const size_t bv = (size_t)d.num_kv_heads * page_bytes_of(d, 1);
  unsigned char* body = const_cast<unsigned char*>(reinterpret_cast<const unsigned char*>(image_body));
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, body) != cudaSuccess) return fail(TQ_ERR_CUDA, "cudaPointerGetAttributes");
  unsigned char* dbody = reinterpret_cast<unsigned char*>(at.devicePointer ? at.devicePointer : body);
  for (int64_t i0 = 0; i0 < n; i0 += kMaxIds) {
    const int cnt = (int)((n - i0) < kMaxIds ? (n - i0) : kMaxIds);
    BlockIds ids;
    std::memcpy(ids.id, blocks + i0, (size_t)cnt * sizeof(int32_t));
    const int grid = cnt < num_sms * 4 ? cnt : num_sms * 4;
    k_copy_blocks<<<grid, 256, 0, st>>>(reinterpret_cast<unsigned char*>(d.k_cache), dbody + (size_t)i0 * bk, ids,
                                        cnt, bk, to_image ? 1 : 0);
    count_launch();
    k_copy_blocks<<<grid, 256, 0, st>>>(reinterpret_cast<unsigned char*>(d.v_cache), dbody + (size_t)n * bk + (size_t)i0 * bv,
                                        ids, cnt, bv, to_image ? 1 : 0);
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "copy blocks: %s", cudaGetErrorString(e));
  }
  return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

size_t tq_image_bytes(const tq_cache_desc* desc, int64_t n_blocks) {
  clear_error();
  if (check_desc(desc, false) != TQ_OK || n_blocks < 0) return 0;
  const size_t per = (size_t)desc->num_kv_heads * (page_bytes_of(*desc, 0) + page_bytes_of(*desc, 1));
  return kHeaderBytes + (size_t)n_blocks * per;
}

tq_status tq_offload_blocks(const tq_cache_desc* desc, const int32_t* blocks, int64_t n, void* image,
                            size_t image_bytes, void* stream) {
  clear_error();
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if ((s = check_blocks(*desc, blocks, n, "tq_offload_blocks")) != TQ_OK) return s;
  if (!image) return fail(TQ_ERR_INVALID_ARG, "tq_offload_blocks: null image");
  const size_t need = tq_image_bytes(desc, n);
  if (image_bytes < need)
    return fail(TQ_ERR_INVALID_ARG, "tq_offload_blocks: image %zu bytes, need %zu", image_bytes, need);
  if ((s = check_image_memory(image, "tq_offload_blocks")) != TQ_OK) return s;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(TQ_ERR_CUDA, "tq_offload_blocks: no device");
  unsigned char* img = reinterpret_cast<unsigned char*>(image);
  make_header(*desc, n, img);
  return copy_blocks(*desc, blocks, n, img + kHeaderBytes, true, sms, reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_restore_blocks(const tq_cache_desc* desc, const int32_t* blocks, int64_t n, const void* image,
                            size_t image_bytes, void* stream) {
  clear_error();
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if ((s = check_blocks(*desc, blocks, n, "tq_restore_blocks")) != TQ_OK) return s;
  if (!image) return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: null image");
  if ((s = check_image_memory(image, "tq_restore_blocks")) != TQ_OK) return s;
  const unsigned char* img = reinterpret_cast<const unsigned char*>(image);
  if (image_bytes < kHeaderBytes || std::memcmp(img, kMagic, 8) != 0)
    return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: not a cache image");
  if (get32(img + 8) != TQ_FORMAT_VERSION)
    return fail(TQ_ERR_VERSION, "tq_restore_blocks: image format version %u, library %u", get32(img + 8),
                TQ_FORMAT_VERSION);
  unsigned char expect[kHeaderBytes];
  make_header(*desc, n, expect);
  if (std::memcmp(img + 12, expect + 12, 36) != 0)
    return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: the image holds another layer format or shape");
  if (get64(img + 48) != (uint64_t)n)
    return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: the image holds %llu blocks, %lld given",
                (unsigned long long)get64(img + 48), (long long)n);
  if (get64(img + 56) != get64(expect + 56))
    return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: the image was made with other codebooks");
  const size_t need = tq_image_bytes(desc, n);
  if (image_bytes < need)
    return fail(TQ_ERR_INVALID_ARG, "tq_restore_blocks: image %zu bytes, need %zu", image_bytes, need);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(TQ_ERR_CUDA, "tq_restore_blocks: no device");
  return copy_blocks(*desc, blocks, n, img + kHeaderBytes, false, sms, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
