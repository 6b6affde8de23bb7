// pa_prefill.cu - causal prefill attention over the paged KV pool on the tcgen05 tensor cores.
//
// Method: PagedAttention summary page, paragraph on the two phases (the prompt phase processes
// all prompt tokens at once as matrix-matrix work and builds their KV cache) and the block
// table; "When KV Capacity Runs Out", Figure 3 (recomputation feeds all retained tokens
// together). Query i of a chunk of n tokens over a cache of L positions stands at position
// L - n + i and attends to positions 0 .. L - n + i.
//
// GB300 design: one CTA per (sequence, kv head, tile of 128 query rows); a row is one (token,
// query head of the group), so a tile holds 128 / G tokens and the GQA group shares every K/V
// tile. K/V tiles of 64 keys stream through a 2-stage shared-memory ring (about 113 KB per CTA
// at head_dim 128, so two CTAs share an SM and overlap each other's softmax and MMA phases):
//   * warps 0 and 2 issue 2-D TMA copies of the K and the V tiles through the block table
//     (copy units of min(block_size, 64) rows, 128-byte swizzle), each through its own ring;
//   * warp 1 allocates tensor memory and one lane issues the MMAs: S_j = Q K_j^T (M 128, N 64)
//     into one of two TMEM S buffers, and O += P_{j-1} V_{j-1} (M 128, N = head_dim) into the
//     TMEM O accumulator, each completion signalled by tcgen05.commit on an mbarrier;
//   * warps 4-7 (one thread per row) read S with tcgen05.ld, apply the causal mask and the
//     online softmax (log2 domain), write P (16-bit, swizzled K-major) to shared memory and
//     rescale O in tensor memory when a row's running maximum grows; at the end they divide O
//     by the row sums and store the output.
// Every wait is bounded; on a timeout the CTA flags PA_ERR_TIMEOUT, drains its MMAs through one
// last commit and frees its tensor memory before it returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kPfThreads = 256;   // 8 warps
constexpr int kPfRows = 128;      // query rows per tile = MMA M
constexpr int kPfKeys = 64;       // keys per K/V tile: S columns, PV reduction
constexpr int kPfStages = 2;      // K/V ring depth (two CTAs fit on an SM)
constexpr int kSoftmaxWarp0 = 4;  // warps 4..7 form the softmax warpgroup
constexpr uint32_t kTmemCols = 256;  // O at columns [0, head_dim), S buffers at [128, 192), [192, 256)

struct PrefillParams {
  const uint16_t* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  const int32_t* q_starts;
  int32_t* err;
  int num_q_heads, num_kv_heads, block_size, log2_block, num_blocks, max_blocks;
  int log2_urows;    // rows per K/V copy: min(block_size, 64)
  float scale_log2;  // scale * log2(e)
};

// 16 fp32 values as 8 packed 16-bit pairs in memory order.
template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack16(uint32_t u) {
  if constexpr (BF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kPfThreads, 2)
    pa_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const __grid_constant__ PrefillParams p) {
  constexpr int kRegions = D / 64;
  constexpr int kTokens = kPfRows / G;
  constexpr uint32_t kQRegion = kPfRows * 128;        // 16 KiB
  constexpr uint32_t kKVRegion = kPfKeys * 128;       // 8 KiB
  constexpr uint32_t kKVBytes = kRegions * kKVRegion;  // K (or V) of one stage

  const int s = blockIdx.z, g = blockIdx.y, t0 = blockIdx.x * kTokens;
  const int q0 = __ldg(p.q_starts + s);
  const int n = __ldg(p.q_starts + s + 1) - q0;
  if (t0 >= n) return;  // the whole CTA: no query of this tile
  const int L = __ldg(p.ctx_lens + s);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_q_heads;

  // invalid lengths (or a chunk longer than the grid's max_q_len): zero rows, flag
  if (n > L || L > p.max_blocks * p.block_size || n > static_cast<int>(gridDim.x) * kTokens) {
    if (tid == 0) flag_error(p.err, kErrCtxLen);
    for (int idx = tid; idx < kPfRows * (D / 8); idx += kPfThreads) {
      const int r = idx / (D / 8), c8 = idx % (D / 8), t = t0 + r / G;
      if (t < n)
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                 (static_cast<size_t>(q0 + t) * Hq + g * G + r % G) * D)[c8] =
            make_uint4(0, 0, 0, 0);
    }
    return;
  }

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  uint8_t* bp = smem_raw;
  if ((base & 1023u) != 0) {  // the swizzled operands need 1024-byte alignment
    if (tid == 0) flag_error(p.err, kErrTimeout);
    return;
  }
  const uint32_t sQ = base;
  const uint32_t sKV = sQ + kRegions * kQRegion;  // stage st: K at sKV + 2 st kKVBytes, V after it
  const uint32_t sP = sKV + kPfStages * 2 * kKVBytes;
  uint8_t* bars_p = bp + (sP - base) + kPfRows * 128;
  // K and V stream through separate rings: K of tile j is free once S_j is computed, V once
  // PV_j is, so K loads run a whole softmax ahead of V loads.
  uint64_t* k_full = reinterpret_cast<uint64_t*>(bars_p);  // [kPfStages]
  uint64_t* k_empty = k_full + kPfStages;                   // [kPfStages]
  uint64_t* v_full = k_empty + kPfStages;                   // [kPfStages]
  uint64_t* v_empty = v_full + kPfStages;                   // [kPfStages]
  uint64_t* s_full = v_empty + kPfStages;                   // [2]
  uint64_t* s_free = s_full + 2;                             // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // causal extent of the tile: its last query stands at position L - n + t_last
  const int t_last = min(n, t0 + kTokens) - 1;
  const int nkeys = L - n + t_last + 1;
  const int ntiles = (nkeys + kPfKeys - 1) / kPfKeys;

  // Q tile -> shared memory, swizzled K-major; rows past the chunk are zero. Every load of a
  // thread is issued before its first store (one memory latency, not one per load), and the
  // loads are in flight while the barriers and tensor memory are set up.
  constexpr int kQLoads = kPfRows * (D / 8) / kPfThreads;  // 16-byte loads per thread
  static_assert(kPfRows * (D / 8) % kPfThreads == 0, "the Q tile splits evenly over the threads");
  uint4 qv[kQLoads];
#pragma unroll
  for (int i = 0; i < kQLoads; ++i) {
    const int idx = tid + i * kPfThreads;
    const int r = idx / (D / 8), c8 = idx % (D / 8), t = t0 + r / G;
    qv[i] = t < n ? __ldg(reinterpret_cast<const uint4*>(
                              p.q + (static_cast<size_t>(q0 + t) * Hq + g * G + r % G) * D) + c8)
                  : make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(smem_addr(k_full + i), 1);
      mbar_init(smem_addr(k_empty + i), 1);
      mbar_init(smem_addr(v_full + i), 1);
      mbar_init(smem_addr(v_empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(s_full + i), 1);
      mbar_init(smem_addr(s_free + i), 4);
    }
    mbar_init(smem_addr(p_full), 4);
    mbar_init(smem_addr(o_done), 1);
    mbar_init(smem_addr(drain), 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
#pragma unroll
  for (int i = 0; i < kQLoads; ++i) {
    const int idx = tid + i * kPfThreads;
    const int r = idx / (D / 8), c8 = idx % (D / 8);
    *reinterpret_cast<uint4*>(bp + (c8 / 8) * kQRegion + sw128_offset(r, c8 % 8)) = qv[i];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem, tS = tmem + 128;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ K/V producers
    // warp 0 streams K, warp 2 streams V, each through its own ring (two lanes of one warp
    // would hold each other up in their barrier waits)
    if (lane == 0) {
      const bool is_v = warp == 2;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      uint64_t* fullb = is_v ? v_full : k_full;
      uint64_t* emptyb = is_v ? v_empty : k_empty;
      const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
      const uint64_t pol = policy_evict_normal();  // the sequence's other query tiles reread them
      const int urows = 1 << p.log2_urows, B = p.block_size;
      const int units = kPfKeys >> p.log2_urows;
      prefetch_tensormap(map);
      // The block-table entries of tile j + 1 are read while the producer waits for a free
      // stage for tile j + 1, so their latency is off the copy path.
      int ph[8];
      auto load_phys = [&](int j) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int key = j * kPfKeys + u * urows;
          ph[u] = (u < units && key < L) ? __ldg(trow + (key >> p.log2_block)) : -2;
        }
      };
      load_phys(0);
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % kPfStages;
        if (j >= kPfStages &&
            !mbar_wait_bounded(smem_addr(emptyb + st), ((j / kPfStages) - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        int rowc[8];
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int key = j * kPfKeys + u * urows;
          rowc[u] = -1;
          if (ph[u] == -2) continue;  // past the unit count or the cache
          if (ph[u] < 0 || ph[u] >= p.num_blocks) {
            if (!is_v) flag_error(p.err, kErrBlockId);
          } else {
            rowc[u] = (ph[u] * p.num_kv_heads + g) * B + (key & (B - 1));
            bytes += static_cast<uint32_t>(kRegions * urows * 128);
          }
        }
        const uint32_t full = smem_addr(fullb + st);
        mbar_arrive_expect_tx(full, bytes);
        const uint32_t dst = sKV + 2 * st * kKVBytes + (is_v ? kKVBytes : 0u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (rowc[u] < 0) continue;
#pragma unroll
          for (int c = 0; c < kRegions; ++c)
            tma_load_2d(dst + c * kKVRegion + static_cast<uint32_t>(u * urows * 128), map, c * 64,
                        rowc[u], full, pol);
        }
        issued = j + 1;
        if (j + 1 < ntiles) load_phys(j + 1);
      }
      // no copy of this CTA may still be landing when it exits (matters after an abort)
      for (int jj = max(0, issued - kPfStages); jj < issued; ++jj)
        mbar_wait_bounded(smem_addr(fullb + jj % kPfStages), (jj / kPfStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_f16(kPfRows, kPfKeys, BF16, false);
      constexpr uint32_t idO = umma_idesc_f16(kPfRows, D, BF16, true);
      // Issue S_ns as soon as K_ns has landed (and its S buffer is free), and PV_npv as soon as
      // P_npv and V_npv are ready, whichever comes first: a late K tile does not hold up the
      // PV of the previous tile. PVs go in tile order (they accumulate into O).
      bool ok = true;
      int ns = 0, npv = 0;
      uint32_t idle = 0;
      unsigned long long idle_since = 0;
      while (npv < ntiles) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        bool did = false;
        if (ns < ntiles) {
          const int st = ns % kPfStages, b = ns & 1;
          if (mbar_test(smem_addr(k_full + st), (ns / kPfStages) & 1) &&
              (ns < 2 || mbar_test(smem_addr(s_free + b), ((ns >> 1) - 1) & 1))) {
            tc_fence_after();
            const uint32_t kst = sKV + 2 * st * kKVBytes;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t c = k / 4, kk = k % 4;
              umma_f16(tS + 64 * b, umma_sdesc(sQ + c * kQRegion + kk * 32, 16, 1024),
                       umma_sdesc(kst + c * kKVRegion + kk * 32, 16, 1024), idS, k > 0);
            }
            umma_commit(smem_addr(s_full + b));
            umma_commit(smem_addr(k_empty + st));
            ++ns;
            did = true;
          }
        }
        if (npv < ns) {
          const int stp = npv % kPfStages;
          if (mbar_test(smem_addr(p_full), npv & 1) &&
              mbar_test(smem_addr(v_full + stp), (npv / kPfStages) & 1)) {
            tc_fence_after();
            const uint32_t vst = sKV + 2 * stp * kKVBytes + kKVBytes;
#pragma unroll
            for (int k = 0; k < kPfKeys / 16; ++k)
              umma_f16(tO, umma_sdesc(sP + k * 32, 16, 1024),
                       umma_sdesc(vst + k * 16 * 128, kKVRegion, 1024), idO, npv > 0 || k > 0);
            umma_commit(smem_addr(o_done));
            umma_commit(smem_addr(v_empty + stp));
            ++npv;
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (idle++ == 0) {
          idle_since = global_ns();
        } else if ((idle & 63u) == 0 && global_ns() - idle_since > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        flag_error(p.err, kErrTimeout);
        *abort_flag = 1;
      }
      // every MMA this thread issued has completed before tensor memory is released
      umma_commit(smem_addr(drain));
      mbar_wait_bounded(smem_addr(drain), 0);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------------ softmax warpgroup
    const int r = tid - kSoftmaxWarp0 * 32;  // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp - kSoftmaxWarp0) * 32) << 16;
    const int tr = t0 + r / G;
    const bool row_valid = tr < n;
    const int pos = L - n + tr;  // last position this row may see
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      ok = mbar_wait_bounded(smem_addr(s_full + b), (j >> 1) & 1);
      if (__any_sync(0xffffffffu, !ok) || *abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kPfKeys];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32_nowait(tS + 64 * b + lane_base, r0);
        tmem_ld32_nowait(tS + 64 * b + lane_base + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[32 + i] = __uint_as_float(r1[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(s_free + b));

      const int key0 = j * kPfKeys;
      // Rows that see all 64 keys of the tile (every tile before the diagonal) need no mask.
      // Scores stay raw until the exponent: m is kept in scaled log2 units and the weight of
      // score x is 2^(x * scale_log2 - m), one FFMA and one ex2.
      const bool full = row_valid && key0 + kPfKeys - 1 <= pos;
      const int lim = row_valid ? pos - key0 : -1;  // last visible column (full: >= 63)
      float mt = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) mt = fmaxf(mt, x[c]);
      } else {
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c)
          if (c <= lim) mt = fmaxf(mt, x[c]);
      }
      mt = mt == -INFINITY ? -INFINITY : mt * p.scale_log2;
      // Lazy rescaling: the row keeps its reference maximum m unless the tile's maximum exceeds
      // it by more than 8 (log2 units); weights then stay below 2^8 and O is rescaled rarely.
      // Numerator and denominator share the same reference, so the result is unchanged.
      const float m_new = mt > m + 8.f ? mt : m;
      const float alpha = m_new == m ? 1.f : ex2(m - m_new);
      uint32_t pk[kPfKeys / 2];
      float psum = 0.f;
      if (full) {
#pragma unroll
        for (int c = 0; c < kPfKeys; c += 2) {
          const float p0 = ex2(fmaf(x[c], p.scale_log2, -m_new));
          const float p1 = ex2(fmaf(x[c + 1], p.scale_log2, -m_new));
          pk[c / 2] = pack16<BF16>(p0, p1);
          psum += p0 + p1;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kPfKeys; c += 2) {
          const float p0 = c <= lim && m_new != -INFINITY ? ex2(fmaf(x[c], p.scale_log2, -m_new)) : 0.f;
          const float p1 =
              c + 1 <= lim && m_new != -INFINITY ? ex2(fmaf(x[c + 1], p.scale_log2, -m_new)) : 0.f;
          pk[c / 2] = pack16<BF16>(p0, p1);
          psum += p0 + p1;
        }
      }
      l = l * alpha + psum;
      m = m_new;

      if (j >= 1) {  // PV_{j-1} done: O is stable and the P buffer free
        ok = mbar_wait_bounded(smem_addr(o_done), (j - 1) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (j == ntiles - 1 && key0 + kPfKeys > L) {
        // value rows past the cache's last position (stale slots, or not loaded) become zero,
        // so that zero weights cannot meet a NaN; the tile's V copies must have landed first
        ok = mbar_wait_bounded(smem_addr(v_full + (j % kPfStages)), (j / kPfStages) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        const uint32_t vst = sKV + 2 * ((ntiles - 1) % kPfStages) * kKVBytes + kKVBytes;
        const int r0 = L - key0;
        const int nbytes16 = (kPfKeys - r0) * 8 * kRegions;  // 16-byte chunks to clear
        for (int i = r; i < nbytes16; i += 128) {
          const int c = i % (8 * kRegions), row = r0 + i / (8 * kRegions);
          *reinterpret_cast<uint4*>(bp + (vst - base) + (c / 8) * kKVRegion + row * 128 +
                                    (c % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // P row r, swizzled K-major: 16-byte chunk c holds keys 8c .. 8c + 7
      uint8_t* prow = bp + (sP - base);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + sw128_offset(r, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {
          float v[16];
          tmem_ld16(tO + lane_base + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= alpha;
          tmem_st16(tO + lane_base + c, v);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(p_full));
    }
    if (ok) ok = mbar_wait_bounded(smem_addr(o_done), (ntiles - 1) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) {
        flag_error(p.err, kErrTimeout);
        *abort_flag = 1;
      }
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                            (static_cast<size_t>(q0 + tr) * Hq + g * G + r % G) * D);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        tmem_ld32_nowait(tO + lane_base + c, v);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack16<BF16>(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[c / 8 + i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }

  // ---- teardown: tensor memory is released once every warp is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

std::mutex& pf_mutex() {
  static std::mutex m;
  return m;
}
std::set<std::pair<const void*, int>>& pf_opted() {
  static std::set<std::pair<const void*, int>> s;
  return s;
}

template <int D, int G, bool BF16>
cudaError_t launch_prefill(const CUtensorMap& km, const CUtensorMap& vm, const PrefillParams& p,
                           dim3 grid, size_t smem, cudaStream_t stream) {
  auto fn = pa_prefill_kernel<D, G, BF16>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(pf_mutex());
    const std::pair<const void*, int> key{reinterpret_cast<const void*>(fn), dev};
    if (!pf_opted().count(key)) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      pf_opted().insert(key);
    }
  }
  fn<<<grid, kPfThreads, smem, stream>>>(km, vm, p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_prefill_g(int group, const CUtensorMap& km, const CUtensorMap& vm,
                             const PrefillParams& p, dim3 grid, size_t smem, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefill<D, 1, BF16>(km, vm, p, grid, smem, stream);
    case 2: return launch_prefill<D, 2, BF16>(km, vm, p, grid, smem, stream);
    case 4: return launch_prefill<D, 4, BF16>(km, vm, p, grid, smem, stream);
    case 8: return launch_prefill<D, 8, BF16>(km, vm, p, grid, smem, stream);
    default: return launch_prefill<D, 16, BF16>(km, vm, p, grid, smem, stream);
  }
}

bool al16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

pa_status run_prefill(const pa_prefill_args& a, cudaStream_t stream, std::string& msg) {
  if (a.num_seqs < 0 || a.num_tokens < 0 || a.max_q_len < 0) {
    msg = "num_seqs, num_tokens and max_q_len must be >= 0";
    return PA_EINVAL;
  }
  if (a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.num_q_heads % a.num_kv_heads != 0) {
    msg = "num_q_heads must be a positive multiple of num_kv_heads";
    return PA_EINVAL;
  }
  const int group = a.num_q_heads / a.num_kv_heads;
  if (a.dtype != PA_F16 && a.dtype != PA_BF16) {
    msg = "pa_prefill supports PA_F16 and PA_BF16";
    return PA_EUNSUPPORTED;
  }
  if (a.head_dim != 64 && a.head_dim != 128) {
    msg = "head_dim must be 64 or 128";
    return PA_EUNSUPPORTED;
  }
  if (a.block_size != 8 && a.block_size != 16 && a.block_size != 32 && a.block_size != 64) {
    msg = "pa_prefill supports block_size 8, 16, 32 or 64";
    return PA_EUNSUPPORTED;
  }
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16) {
    msg = "group size must be 1, 2, 4, 8 or 16";
    return PA_EUNSUPPORTED;
  }
  if (a.num_blocks <= 0 || a.max_blocks_per_seq <= 0) {
    msg = "num_blocks and max_blocks_per_seq must be positive";
    return PA_EINVAL;
  }
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * a.block_size;
  if (rows >= (1ll << 31)) {
    msg = "pool has more than 2^31 token rows";
    return PA_EUNSUPPORTED;
  }
  if (a.num_seqs == 0 || a.num_tokens == 0 || a.max_q_len == 0) return PA_OK;
  if (!a.q || !a.k_pool || !a.v_pool || !a.block_tables || !a.ctx_lens || !a.q_starts || !a.out) {
    msg = "null pointer argument";
    return PA_EINVAL;
  }
  if (!al16(a.q) || !al16(a.out) || !al16(a.k_pool) || !al16(a.v_pool)) {
    msg = "q, out and the pools must be 16-byte aligned";
    return PA_EINVAL;
  }
  const int urows = std::min(a.block_size, kPfKeys);
  CUtensorMap kmap, vmap;
  pa_status st = encode_pool_rows_map(&kmap, a.k_pool, rows, a.head_dim, 2, urows, msg);
  if (st != PA_OK) return st;
  st = encode_pool_rows_map(&vmap, a.v_pool, rows, a.head_dim, 2, urows, msg);
  if (st != PA_OK) return st;

  PrefillParams p{};
  p.q = static_cast<const uint16_t*>(a.q);
  p.out = a.out;
  p.err = a.err_flag;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.log2_block = 0;
  while ((1 << p.log2_block) < a.block_size) ++p.log2_block;
  p.log2_urows = 0;
  while ((1 << p.log2_urows) < urows) ++p.log2_urows;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks_per_seq;
  p.scale_log2 = a.scale * 1.4426950408889634f;

  const int D = a.head_dim;
  const size_t regions = static_cast<size_t>(D / 64);
  // no alignment slack: the kernel needs (and checks) a 1024-byte aligned dynamic region, and
  // two CTAs then fit on an SM
  const size_t smem = regions * kPfRows * 128 + kPfStages * 2 * regions * kPfKeys * 128 +
                      kPfRows * 128 + 256;
  const int tokens_per_tile = kPfRows / group;
  const unsigned tiles = static_cast<unsigned>((a.max_q_len + tokens_per_tile - 1) / tokens_per_tile);
  const bool bf16 = a.dtype == PA_BF16;
  constexpr int kMaxZ = 65535;
  for (int s0 = 0; s0 < a.num_seqs; s0 += kMaxZ) {
    const int ns = std::min(kMaxZ, a.num_seqs - s0);
    p.block_tables = a.block_tables + static_cast<size_t>(s0) * a.max_blocks_per_seq;
    p.ctx_lens = a.ctx_lens + s0;
    p.q_starts = a.q_starts + s0;
    const dim3 grid(tiles, static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(ns));
    cudaError_t e;
    if (D == 128)
      e = bf16 ? launch_prefill_g<128, true>(group, kmap, vmap, p, grid, smem, stream)
               : launch_prefill_g<128, false>(group, kmap, vmap, p, grid, smem, stream);
    else
      e = bf16 ? launch_prefill_g<64, true>(group, kmap, vmap, p, grid, smem, stream)
               : launch_prefill_g<64, false>(group, kmap, vmap, p, grid, smem, stream);
    st = cuda_status(e, "pa_prefill kernel launch", msg);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

}  // namespace pa
