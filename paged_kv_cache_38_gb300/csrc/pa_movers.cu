// pa_movers.cu - block data movers: write-KV scatter, copy-on-write block copy, swap out/in.
//
// Sources: "When KV Capacity Runs Out: Pausing and Resuming Requests", Figure 2 (the KV of a
// newly processed position goes into its slot) and Figure 4 (a preempted request's KV is copied
// to CPU memory and later restored, possibly into other blocks); "Efficient Memory Management
// for Large Language Model Serving with PagedAttention" (summary page), paragraph on
// copy-on-write; "KV Cache Preemption in vLLM", section "Swap versus recompute" (pinned memory,
// a block's data is spread over every layer, so a swap moves 2 * layers slabs per block).
//
// All three are byte moves: 16-byte vector loads and stores, several in flight per thread. The
// quantise-on-write variant of the write ("KV Cache Preemption in vLLM", section "How much KV
// cache a token costs": an FP8 cache holds one byte per element) converts on the way.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kMaxLayers = 256;
constexpr int kMaxIdsPerLaunch = 2048;
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte vectors per thread per step
constexpr int kSliceBytes = kCopyThreads * kCopyUnroll * 16;  // 16 KiB per CTA step

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ write-KV

struct WriteParams {
  const uint4* k;
  const uint4* v;
  uint4* k_pool;
  uint4* v_pool;
  const int64_t* slots;
  int32_t* err;
  int num_tokens, num_kv_heads, chunks_per_row, block_size, num_blocks;
  int log2_chunks, log2_block;  // when chunks_per_row and block_size are powers of two
};

// pool[slot/B][h][slot%B][:] = new[t][h][:], in 16-byte chunks of (token, kv head) rows. Each
// thread moves two chunks per pass, both loads issued before either store; the loads do not wait
// for the slot, only the stores do. Index arithmetic is 32-bit (the host keeps a launch below
// 2^31 chunks), with shifts when the row's chunk count and the block size are powers of two.
template <bool kPow2>
__global__ void __launch_bounds__(256) pa_write_kv_kernel(const __grid_constant__ WriteParams p) {
  const uint32_t total = static_cast<uint32_t>(p.num_tokens) * p.num_kv_heads * p.chunks_per_row;
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t H = p.num_kv_heads, cpr = p.chunks_per_row, B = p.block_size;
  for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    uint4 kk[2], vv[2];
    uint32_t th[2], c[2];
    bool in[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t i = i0 + u * stride;
      in[u] = i < total;
      c[u] = kPow2 ? (i & (cpr - 1)) : i % cpr;
      th[u] = kPow2 ? (i >> p.log2_chunks) : i / cpr;
      if (in[u]) {
        const size_t src = static_cast<size_t>(th[u]) * cpr + c[u];
        kk[u] = __ldg(p.k + src);
        vv[u] = __ldg(p.v + src);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!in[u]) continue;
      const uint32_t t = th[u] / H, h = th[u] - t * H;
      const long long slot = __ldg(p.slots + t);
      if (slot < 0) continue;  // padding token
      const long long blk = kPow2 ? (slot >> p.log2_block) : slot / B;
      if (blk >= p.num_blocks) {
        if (h == 0 && c[u] == 0) flag_error(p.err, kErrBlockId);
        continue;
      }
      const long long off = kPow2 ? (slot & (B - 1)) : slot % B;
      const size_t dst = ((static_cast<size_t>(blk) * H + h) * B + off) * cpr + c[u];
      p.k_pool[dst] = kk[u];
      p.v_pool[dst] = vv[u];
    }
  }
}

int log2_exact(int x) { return x > 0 && (x & (x - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(x)) : -1; }

// ------------------------------------------------------------------ quantise-on-write (E4M3)

struct WriteFp8Params {
  const uint4* k;   // 16-bit rows: two 16-byte vectors per chunk of 16 elements
  const uint4* v;
  uint4* k_pool;    // E4M3 rows: one 16-byte vector per chunk
  uint4* v_pool;
  const int64_t* slots;
  int32_t* err;
  float k_scale, v_scale;
  int src_bf16;
  int num_tokens, num_kv_heads, chunks_per_row, block_size, num_blocks;
  int log2_chunks, log2_block;  // when chunks_per_row and block_size are powers of two
};

// Two binary32 values to two E4M3 codes, nearest / ties-to-even, saturating to +-448 (NaN stays
// NaN); `first` lands in the low byte, which comes first in memory.
__device__ __forceinline__ uint32_t e4m3x2(float first, float second) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

// Eight 16-bit values (one 16-byte vector) times rcp = RN(1 / scale), rounded to binary32, as
// eight E4M3 codes.
__device__ __forceinline__ uint2 quantise8(uint4 w, float rcp, bool bf16) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      f[2 * i] = __uint_as_float(words[i] << 16);
      f[2 * i + 1] = __uint_as_float(words[i] & 0xffff0000u);
    } else {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&words[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) pk[i] = e4m3x2(__fmul_rn(f[2 * i], rcp), __fmul_rn(f[2 * i + 1], rcp));
  uint2 r;
  r.x = pk[0] | (pk[1] << 16);
  r.y = pk[2] | (pk[3] << 16);
  return r;
}

// Each thread converts two 16-element chunks of (token, kv head) rows per pass, both chunks'
// loads issued before either is converted; the loads do not wait for the slot, only the stores
// do. Index arithmetic is 32-bit (the host keeps a launch below 2^31 chunks), with shifts when
// the row's chunk count and the block size are powers of two.
template <bool kPow2>
__global__ void __launch_bounds__(256) pa_write_kv_fp8_kernel(const __grid_constant__ WriteFp8Params p) {
  const uint32_t total = static_cast<uint32_t>(p.num_tokens) * p.num_kv_heads * p.chunks_per_row;
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t H = p.num_kv_heads, cpr = p.chunks_per_row, B = p.block_size;
  const bool bf16 = p.src_bf16 != 0;
  const float k_rcp = __frcp_rn(p.k_scale), v_rcp = __frcp_rn(p.v_scale);  // IEEE reciprocals
  for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    uint4 kk[2][2], vv[2][2];
    uint32_t th[2], c[2];
    bool in[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t i = i0 + u * stride;
      in[u] = i < total;
      c[u] = kPow2 ? (i & (cpr - 1)) : i % cpr;
      th[u] = kPow2 ? (i >> p.log2_chunks) : i / cpr;
      if (in[u]) {
        const size_t src = 2 * (static_cast<size_t>(th[u]) * cpr + c[u]);
        kk[u][0] = __ldg(p.k + src);
        kk[u][1] = __ldg(p.k + src + 1);
        vv[u][0] = __ldg(p.v + src);
        vv[u][1] = __ldg(p.v + src + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!in[u]) continue;
      const uint32_t t = th[u] / H, h = th[u] - t * H;
      const long long slot = __ldg(p.slots + t);
      if (slot < 0) continue;  // padding token
      const long long blk = kPow2 ? (slot >> p.log2_block) : slot / B;
      if (blk >= p.num_blocks) {
        if (h == 0 && c[u] == 0) flag_error(p.err, kErrBlockId);
        continue;
      }
      const long long off = kPow2 ? (slot & (B - 1)) : slot % B;
      const size_t dst = ((static_cast<size_t>(blk) * H + h) * B + off) * cpr + c[u];
      const uint2 kq0 = quantise8(kk[u][0], k_rcp, bf16), kq1 = quantise8(kk[u][1], k_rcp, bf16);
      const uint2 vq0 = quantise8(vv[u][0], v_rcp, bf16), vq1 = quantise8(vv[u][1], v_rcp, bf16);
      p.k_pool[dst] = make_uint4(kq0.x, kq0.y, kq1.x, kq1.y);
      p.v_pool[dst] = make_uint4(vq0.x, vq0.y, vq1.x, vq1.y);
    }
  }
}

// ------------------------------------------------------------------ region copies

// kCopyPairs: device (src, dst) pairs. kPoolToBuf / kBufToPool: entry i is block ids[i] and
// buffer slot i. kHostPairs: (src, dst) pairs in ids. kPoolToSlots: (block, buffer slot) pairs in
// ids; kSlotsToPool: (buffer slot, block) pairs in ids (a plan's swap lists).
enum CopyMode { kCopyPairs = 0, kPoolToBuf = 1, kBufToPool = 2, kHostPairs = 3, kPoolToSlots = 4,
                kSlotsToPool = 5 };

struct CopyParams {
  uint8_t* k[kMaxLayers];
  uint8_t* v[kMaxLayers];
  uint8_t* buf;          // host-mapped pinned buffer or device staging, [slots][layers][2][bytes]
  const int32_t* pairs;  // kCopyPairs: device [n][2]
  int32_t* err;
  int32_t ids[kMaxIdsPerLaunch];  // block ids, or id pairs, of this launch (host-validated)
  long long block_bytes;
  int mode, n, num_layers, num_blocks, slices_per_region;
};

// Region r = ((i * layers) + l) * 2 + kv moves one (block, layer, K|V) slab of block_bytes.
// Work unit = one 16 KiB slice of a region; each thread keeps 4 x 16 bytes in flight.
__global__ void __launch_bounds__(kCopyThreads) pa_copy_regions_kernel(const __grid_constant__ CopyParams p) {
  const long long regions = static_cast<long long>(p.n) * p.num_layers * 2;
  const long long units = regions * p.slices_per_region;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long r = u / p.slices_per_region;
    const int slice = static_cast<int>(u % p.slices_per_region);
    const int kv = static_cast<int>(r & 1);
    const int l = static_cast<int>((r >> 1) % p.num_layers);
    const int i = static_cast<int>((r >> 1) / p.num_layers);
    const uint8_t* src;
    uint8_t* dst;
    uint8_t* pool = kv ? p.v[l] : p.k[l];
    if (p.mode == kCopyPairs || p.mode == kHostPairs) {
      int s, d;
      if (p.mode == kCopyPairs) {
        s = __ldg(p.pairs + 2 * i);
        d = __ldg(p.pairs + 2 * i + 1);
      } else {
        s = p.ids[2 * i];
        d = p.ids[2 * i + 1];
      }
      if (s < 0 || s >= p.num_blocks || d < 0 || d >= p.num_blocks) {
        if (threadIdx.x == 0 && slice == 0 && l == 0 && kv == 0) flag_error(p.err, kErrBlockId);
        continue;
      }
      src = pool + s * p.block_bytes;
      dst = pool + d * p.block_bytes;
    } else {
      long long blk = p.ids[i], slot = i;
      if (p.mode == kPoolToSlots) {
        blk = p.ids[2 * i];
        slot = p.ids[2 * i + 1];
      } else if (p.mode == kSlotsToPool) {
        slot = p.ids[2 * i];
        blk = p.ids[2 * i + 1];
      }
      uint8_t* slab = pool + blk * p.block_bytes;
      uint8_t* packed = p.buf + ((slot * p.num_layers + l) * 2 + kv) * p.block_bytes;
      const bool out = p.mode == kPoolToBuf || p.mode == kPoolToSlots;
      src = out ? slab : packed;
      dst = out ? packed : slab;
    }
    const long long off0 = static_cast<long long>(slice) * kSliceBytes;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + off0);
    uint4* d4 = reinterpret_cast<uint4*>(dst + off0);
    const long long left = (p.block_bytes - off0) / 16;  // vectors remaining in this region
    uint4 tmp[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) {
      const long long idx = threadIdx.x + static_cast<long long>(k) * kCopyThreads;
      if (idx < left) tmp[k] = s4[idx];
    }
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) {
      const long long idx = threadIdx.x + static_cast<long long>(k) * kCopyThreads;
      if (idx < left) d4[idx] = tmp[k];
    }
  }
}

int copy_grid(long long units) {
  const int sms = std::max(1, device_sm_count());
  return static_cast<int>(std::max(1LL, std::min(units, static_cast<long long>(sms) * 16)));
}

pa_status check_pools(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                      size_t block_bytes, int32_t num_blocks, std::string& msg) {
  if (num_layers <= 0 || num_layers > kMaxLayers) {
    msg = "num_layers must be in [1, 256]";
    return PA_EINVAL;
  }
  if (!k_pools || !v_pools) {
    msg = "null pool array";
    return PA_EINVAL;
  }
  if (block_bytes == 0 || block_bytes % 16 != 0) {
    msg = "block_bytes must be a positive multiple of 16";
    return PA_EINVAL;
  }
  if (num_blocks <= 0) {
    msg = "num_blocks must be positive";
    return PA_EINVAL;
  }
  for (int l = 0; l < num_layers; ++l) {
    if (!k_pools[l] || !v_pools[l] || !aligned16(k_pools[l]) || !aligned16(v_pools[l])) {
      msg = "pool pointer " + std::to_string(l) + " is null or not 16-byte aligned";
      return PA_EINVAL;
    }
  }
  return PA_OK;
}

void fill_pools(CopyParams& p, void* const* k_pools, void* const* v_pools, int32_t num_layers) {
  for (int l = 0; l < num_layers; ++l) {
    p.k[l] = static_cast<uint8_t*>(k_pools[l]);
    p.v[l] = static_cast<uint8_t*>(v_pools[l]);
  }
}

}  // namespace

pa_status run_write_kv(const void* k, const void* v, void* k_pool, void* v_pool,
                       const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype kv_dtype,
                       int32_t* err_flag, cudaStream_t stream, std::string& msg) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0) {
    msg = "sizes must be positive (num_tokens may be 0)";
    return PA_EINVAL;
  }
  if (kv_dtype != PA_F16 && kv_dtype != PA_BF16 && kv_dtype != PA_FP8_E4M3) {
    msg = "unknown kv_dtype";
    return PA_EINVAL;
  }
  const int elt = kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  if ((head_dim * elt) % 16 != 0) {
    msg = "head_dim * element size must be a multiple of 16 bytes";
    return PA_EINVAL;
  }
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) {
    msg = "null pointer argument";
    return PA_EINVAL;
  }
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) {
    msg = "k, v and the pools must be 16-byte aligned, slot_mapping 8-byte aligned";
    return PA_EINVAL;
  }
  WriteParams p{};
  p.k = static_cast<const uint4*>(k);
  p.v = static_cast<const uint4*>(v);
  p.k_pool = static_cast<uint4*>(k_pool);
  p.v_pool = static_cast<uint4*>(v_pool);
  p.slots = slot_mapping;
  p.err = err_flag;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.chunks_per_row = head_dim * elt / 16;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.log2_chunks = log2_exact(p.chunks_per_row);
  p.log2_block = log2_exact(block_size);
  const bool pow2 = p.log2_chunks >= 0 && p.log2_block >= 0;
  // launches of fewer than 2^31 chunks each (32-bit index arithmetic in the kernel)
  const long long row_chunks = static_cast<long long>(num_kv_heads) * p.chunks_per_row;
  const int max_tokens = static_cast<int>(std::max<long long>(1, ((1LL << 31) - 1) / row_chunks));
  for (int t0 = 0; t0 < num_tokens; t0 += max_tokens) {
    WriteParams q = p;
    q.num_tokens = std::min(max_tokens, num_tokens - t0);
    q.k = p.k + static_cast<size_t>(t0) * row_chunks;
    q.v = p.v + static_cast<size_t>(t0) * row_chunks;
    q.slots = p.slots + t0;
    const long long total = static_cast<long long>(q.num_tokens) * row_chunks;
    const int grid = static_cast<int>(std::min<long long>((total + 511) / 512,
                                                          std::max(1, device_sm_count()) * 8LL));
    if (pow2) {
      pa_write_kv_kernel<true><<<grid, 256, 0, stream>>>(q);
    } else {
      pa_write_kv_kernel<false><<<grid, 256, 0, stream>>>(q);
    }
    const pa_status st = cuda_status(cudaGetLastError(), "pa_write_kv launch", msg);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

pa_status run_write_kv_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_pool,
                           void* v_pool, const int64_t* slot_mapping, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t num_blocks, float k_scale, float v_scale, int32_t* err_flag,
                           cudaStream_t stream, std::string& msg) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0) {
    msg = "sizes must be positive (num_tokens may be 0)";
    return PA_EINVAL;
  }
  if (src_dtype != PA_F16 && src_dtype != PA_BF16) {
    msg = "src_dtype must be PA_F16 or PA_BF16";
    return PA_EINVAL;
  }
  if (head_dim % 16 != 0) {
    msg = "head_dim must be a multiple of 16";
    return PA_EINVAL;
  }
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) {
    msg = "k_scale and v_scale must be finite and > 0";
    return PA_EINVAL;
  }
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) {
    msg = "null pointer argument";
    return PA_EINVAL;
  }
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) {
    msg = "k, v and the pools must be 16-byte aligned, slot_mapping 8-byte aligned";
    return PA_EINVAL;
  }
  WriteFp8Params p{};
  p.k = static_cast<const uint4*>(k);
  p.v = static_cast<const uint4*>(v);
  p.k_pool = static_cast<uint4*>(k_pool);
  p.v_pool = static_cast<uint4*>(v_pool);
  p.slots = slot_mapping;
  p.err = err_flag;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.src_bf16 = src_dtype == PA_BF16 ? 1 : 0;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.chunks_per_row = head_dim / 16;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.log2_chunks = log2_exact(p.chunks_per_row);
  p.log2_block = log2_exact(block_size);
  const bool pow2 = p.log2_chunks >= 0 && p.log2_block >= 0;
  // launches of fewer than 2^31 chunks each (32-bit index arithmetic in the kernel)
  const long long row_chunks = static_cast<long long>(num_kv_heads) * p.chunks_per_row;
  const int max_tokens = static_cast<int>(std::max<long long>(1, ((1LL << 31) - 1) / row_chunks));
  for (int t0 = 0; t0 < num_tokens; t0 += max_tokens) {
    WriteFp8Params q = p;
    q.num_tokens = std::min(max_tokens, num_tokens - t0);
    q.k = p.k + 2 * static_cast<size_t>(t0) * row_chunks;
    q.v = p.v + 2 * static_cast<size_t>(t0) * row_chunks;
    q.slots = p.slots + t0;
    const long long total = static_cast<long long>(q.num_tokens) * row_chunks;
    const int grid = static_cast<int>(std::min<long long>((total + 511) / 512,
                                                          std::max(1, device_sm_count()) * 8LL));
    if (pow2) {
      pa_write_kv_fp8_kernel<true><<<grid, 256, 0, stream>>>(q);
    } else {
      pa_write_kv_fp8_kernel<false><<<grid, 256, 0, stream>>>(q);
    }
    const pa_status st = cuda_status(cudaGetLastError(), "pa_write_kv_fp8 launch", msg);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

pa_status run_copy_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                          const int32_t* pairs, int32_t num_pairs, int32_t num_blocks,
                          size_t block_bytes, int32_t* err_flag, cudaStream_t stream,
                          std::string& msg) {
  pa_status st = check_pools(k_pools, v_pools, num_layers, block_bytes, num_blocks, msg);
  if (st != PA_OK) return st;
  if (num_pairs < 0) {
    msg = "num_pairs must be >= 0";
    return PA_EINVAL;
  }
  if (num_pairs == 0) return PA_OK;
  if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 3u)) {
    msg = "pairs must be a 4-byte aligned device pointer";
    return PA_EINVAL;
  }
  CopyParams* p = new CopyParams();
  fill_pools(*p, k_pools, v_pools, num_layers);
  p->pairs = pairs;
  p->err = err_flag;
  p->block_bytes = static_cast<long long>(block_bytes);
  p->mode = kCopyPairs;
  p->n = num_pairs;
  p->num_layers = num_layers;
  p->num_blocks = num_blocks;
  p->slices_per_region = static_cast<int>((block_bytes + kSliceBytes - 1) / kSliceBytes);
  const long long units = static_cast<long long>(num_pairs) * num_layers * 2 * p->slices_per_region;
  pa_copy_regions_kernel<<<copy_grid(units), kCopyThreads, 0, stream>>>(*p);
  delete p;
  return cuda_status(cudaGetLastError(), "pa_copy_blocks launch", msg);
}

pa_status run_swap_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                          void* host_buf, const int32_t* block_ids, int32_t n, int32_t num_blocks,
                          size_t block_bytes, pa_swap_dir dir, void* staging, size_t staging_bytes,
                          cudaStream_t stream, std::string& msg) {
  pa_status st = check_pools(k_pools, v_pools, num_layers, block_bytes, num_blocks, msg);
  if (st != PA_OK) return st;
  if (dir != PA_SWAP_OUT && dir != PA_SWAP_IN) {
    msg = "dir must be PA_SWAP_OUT or PA_SWAP_IN";
    return PA_EINVAL;
  }
  if (n < 0) {
    msg = "n must be >= 0";
    return PA_EINVAL;
  }
  if (n == 0) return PA_OK;
  if (!host_buf || !block_ids || !aligned16(host_buf)) {
    msg = "host_buf (16-byte aligned) and block_ids are required";
    return PA_EINVAL;
  }
  for (int i = 0; i < n; ++i) {
    if (block_ids[i] < 0 || block_ids[i] >= num_blocks) {
      msg = "block_ids[" + std::to_string(i) + "] is outside the pool";
      return PA_EINVAL;
    }
  }
  const size_t total = static_cast<size_t>(n) * num_layers * 2 * block_bytes;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, host_buf) != cudaSuccess) {
    cudaGetLastError();
    msg = "host_buf is not known to CUDA";
    return PA_EINVAL;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
    msg = "host_buf must be pinned host memory (cudaHostAlloc / cudaHostRegister)";
    return PA_EINVAL;
  }
  if (staging != nullptr && (staging_bytes < total || !aligned16(staging))) {
    msg = "staging must hold n * num_layers * 2 * block_bytes bytes, 16-byte aligned";
    return PA_EINVAL;
  }
  uint8_t* mapped = static_cast<uint8_t*>(attr.devicePointer);

  if (staging != nullptr && dir == PA_SWAP_IN) {
    st = cuda_status(cudaMemcpyAsync(staging, host_buf, total, cudaMemcpyHostToDevice, stream),
                     "pa_swap_blocks host-to-device copy", msg);
    if (st != PA_OK) return st;
  }
  CopyParams* p = new CopyParams();
  fill_pools(*p, k_pools, v_pools, num_layers);
  p->block_bytes = static_cast<long long>(block_bytes);
  p->mode = dir == PA_SWAP_OUT ? kPoolToBuf : kBufToPool;
  p->num_layers = num_layers;
  p->num_blocks = num_blocks;
  p->slices_per_region = static_cast<int>((block_bytes + kSliceBytes - 1) / kSliceBytes);
  const size_t per_block = static_cast<size_t>(num_layers) * 2 * block_bytes;
  uint8_t* buf = staging != nullptr ? static_cast<uint8_t*>(staging) : mapped;
  for (int i0 = 0; i0 < n && st == PA_OK; i0 += kMaxIdsPerLaunch) {
    const int cnt = std::min(kMaxIdsPerLaunch, n - i0);
    std::memcpy(p->ids, block_ids + i0, sizeof(int32_t) * cnt);
    p->n = cnt;
    p->buf = buf + static_cast<size_t>(i0) * per_block;
    const long long units = static_cast<long long>(cnt) * num_layers * 2 * p->slices_per_region;
    pa_copy_regions_kernel<<<copy_grid(units), kCopyThreads, 0, stream>>>(*p);
    st = cuda_status(cudaGetLastError(), "pa_swap_blocks launch", msg);
  }
  delete p;
  if (st != PA_OK) return st;
  if (staging != nullptr && dir == PA_SWAP_OUT) {
    st = cuda_status(cudaMemcpyAsync(host_buf, staging, total, cudaMemcpyDeviceToHost, stream),
                     "pa_swap_blocks device-to-host copy", msg);
  }
  return st;
}

pa_status run_plan_moves(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         int32_t num_blocks, size_t block_bytes, void* cpu_pool,
                         int32_t num_cpu_blocks, const int32_t* swap_out, int32_t num_swap_out,
                         const int32_t* swap_in, int32_t num_swap_in, const int32_t* copies,
                         int32_t num_copies, int32_t* err_flag, cudaStream_t stream,
                         std::string& msg) {
  pa_status st = check_pools(k_pools, v_pools, num_layers, block_bytes, num_blocks, msg);
  if (st != PA_OK) return st;
  if (num_swap_out < 0 || num_swap_in < 0 || num_copies < 0 || num_cpu_blocks < 0) {
    msg = "move counts and num_cpu_blocks must be >= 0";
    return PA_EINVAL;
  }
  if ((num_swap_out && !swap_out) || (num_swap_in && !swap_in) || (num_copies && !copies)) {
    msg = "a non-empty move list is NULL";
    return PA_EINVAL;
  }
  // every id is known on the host: check them all before anything is enqueued
  auto check = [&](const int32_t* pairs, int n, int col_slot, const char* what) -> bool {
    for (int i = 0; i < n; ++i) {
      for (int c = 0; c < 2; ++c) {
        const int32_t v = pairs[2 * i + c];
        const int32_t limit = c == col_slot ? num_cpu_blocks : num_blocks;
        if (v < 0 || v >= limit) {
          msg = std::string(what) + "[" + std::to_string(i) + "][" + std::to_string(c) +
                "] = " + std::to_string(v) + " is outside " +
                (c == col_slot ? "the CPU pool" : "the GPU pool");
          return false;
        }
      }
    }
    return true;
  };
  if (!check(swap_out, num_swap_out, 1, "swap_out") || !check(swap_in, num_swap_in, 0, "swap_in") ||
      !check(copies, num_copies, -1, "copies"))
    return PA_EINVAL;
  uint8_t* mapped = nullptr;
  if (num_swap_out + num_swap_in > 0) {
    if (!cpu_pool || !aligned16(cpu_pool)) {
      msg = "cpu_pool (16-byte aligned pinned memory) is required for swaps";
      return PA_EINVAL;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, cpu_pool) != cudaSuccess) {
      cudaGetLastError();
      msg = "cpu_pool is not known to CUDA";
      return PA_EINVAL;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
      msg = "cpu_pool must be pinned host memory (cudaHostAlloc / cudaHostRegister)";
      return PA_EINVAL;
    }
    mapped = static_cast<uint8_t*>(attr.devicePointer);
  }
  CopyParams* p = new CopyParams();
  fill_pools(*p, k_pools, v_pools, num_layers);
  p->buf = mapped;
  p->err = err_flag;
  p->block_bytes = static_cast<long long>(block_bytes);
  p->num_layers = num_layers;
  p->num_blocks = num_blocks;
  p->slices_per_region = static_cast<int>((block_bytes + kSliceBytes - 1) / kSliceBytes);
  // swap-outs, then swap-ins, then copy-on-write copies, in stream order
  const struct {
    const int32_t* pairs;
    int n;
    int mode;
    const char* what;
  } lists[3] = {{swap_out, num_swap_out, kPoolToSlots, "swap-out"},
                {swap_in, num_swap_in, kSlotsToPool, "swap-in"},
                {copies, num_copies, kHostPairs, "copy-on-write"}};
  constexpr int kPairsPerLaunch = kMaxIdsPerLaunch / 2;
  for (const auto& m : lists) {
    for (int i0 = 0; i0 < m.n && st == PA_OK; i0 += kPairsPerLaunch) {
      const int cnt = std::min(kPairsPerLaunch, m.n - i0);
      std::memcpy(p->ids, m.pairs + 2 * i0, sizeof(int32_t) * 2 * cnt);
      p->mode = m.mode;
      p->n = cnt;
      const long long units = static_cast<long long>(cnt) * num_layers * 2 * p->slices_per_region;
      pa_copy_regions_kernel<<<copy_grid(units), kCopyThreads, 0, stream>>>(*p);
      st = cuda_status(cudaGetLastError(), m.what, msg);
    }
  }
  delete p;
  return st;
}

}  // namespace pa
