// pa_prefill.cu - causal prefill attention over the paged KV pool on the tcgen05 tensor cores.
//
// Method: PagedAttention summary page, paragraph on the two phases (the prompt phase processes
// all prompt tokens at once as matrix-matrix work and builds their KV cache) and the block
// table; "When KV Capacity Runs Out", Figure 3 (recomputation feeds all retained tokens
// together). Query i of a chunk of n tokens over a cache of L positions stands at position
// L - n + i and attends to positions 0 .. L - n + i.
//
// GB300 design: a persistent kernel, two CTAs per SM (about 97 KB of shared memory and 256
// tensor-memory columns each at head_dim 128, so the two overlap each other's softmax and MMA
// phases). A work item is one tile of 128 query rows of one (sequence, kv head); a row is one
// (token, query head of the group), so a tile holds 128 / G tokens and the GQA group shares
// every K/V tile. Items are taken from a work counter (or round-robin) in blocks of kTileBlock
// query tiles: the kTileBlock longest tiles of every (sequence, kv head), then the next
// kTileBlock, and so on, so that the batch runs roughly longest first while the pairs in flight
// keep their K/V in L2. Tensor memory, barriers and the K/V rings live across items, so the
// next item's queries and first K/V tiles load while the current one finishes. Roles:
//   * warp 3 takes items and publishes them through a 2-slot ring; it loads each item's query
//     tile (one 3-D TMA box per 64 columns) once the previous item's last S MMA has completed;
//   * warps 0 and 2 issue 2-D TMA copies of the K and the V tiles (64 keys) through the block
//     table (copy units of min(block_size, 64) rows, 128-byte swizzle), each through its own
//     2-stage ring;
//   * warp 1 allocates tensor memory and one lane issues the MMAs: S_j = Q K_j^T (M 128, N 64)
//     into one of two TMEM S buffers, and O += P_j V_j (M 128, N = head_dim) into the TMEM O
//     accumulator with P_j read from tensor memory, PV first when both are ready; one
//     tcgen05.commit per MMA group signals its completion on an mbarrier, which also hands the
//     group's K (or V) stage back to its producer;
//   * warps 4-7 (one thread per row) read S with tcgen05.ld, apply the causal mask and the
//     online softmax (log2 domain, packed fp32 pairs), write P (16-bit pairs) with tcgen05.st
//     over the first half of the S buffer it came from, and rescale O in tensor memory when a
//     row's running maximum grows. P_j thus never waits for PV_{j-1}; only a rescale and the
//     item epilogue read O. An item's epilogue (O divided by the row sums, rows stored) runs
//     inside the next item's first tile, once that tile's P is written, so that the wait for
//     the item's last PV overlaps the next tile's softmax.
// An E4M3 cache (head_dim 128) goes through the same pipeline on f16 MMAs: each K/V copy brings
// the tile's raw bytes into the upper half of its stage and the whole producer warp widens them
// to f16 in place (exact); the query-loader warp moves bf16 query rows to f16, each with a
// power-of-two scale that the softmax folds into its score scale; v_scale joins the epilogue.
// Every wait is bounded (pa_testing_set_wait_limit can shorten the waits of one role on another
// and make one CTA's MMA issuer stop, for tests); on a timeout the CTA flags PA_ERR_TIMEOUT, the
// roles wind down, the copies and MMAs in flight drain (those waits keep a one-second limit)
// and the tensor memory is freed before the CTA returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
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
constexpr int kSlots = 2;         // published work items
constexpr int kTileBlock = 4;     // query tiles of one (sequence, kv head) per block of the order
constexpr int kSoftmaxWarp0 = 4;  // warps 4..7 form the softmax warpgroup
constexpr int kItemReaders = 3 + 4;  // K producer, V producer, MMA issuer, 4 softmax warps
constexpr uint32_t kTmemCols = 256;  // O at columns [0, head_dim), S buffers at [128, 192), [192, 256)
constexpr uint32_t kCtlBytes = 384;  // barriers, item slots, tensor-memory address, abort flag
// the E4M3 cache adds the raw-copy barriers, the per-slot query barriers and the per-row query
// exponents of both item slots
constexpr uint32_t kCtlBytesFp8 = 640;

// Element type of the K/V pools.
enum PfKv { kPfF16 = 0, kPfBF16 = 1, kPfE4M3 = 2 };

// Softmax arithmetic on full tiles: 3-input maxima and packed fp32 pairs (fma / add .f32x2)
// halve the instruction count of the row maximum, the exponent arguments and the row sum; the
// softmax warps share their schedulers with the other CTA's and are bound by issue.
// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// two fp32 lanes in one 64-bit register pair
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// (a * b + c) per lane, rounded once (the same result as two fmaf)
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

struct PrefillParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  const int32_t* q_starts;
  int32_t* err;
  int32_t* work;  // work counter, or null for round-robin items
  int num_tokens, num_q_heads, num_kv_heads, block_size, log2_block, num_blocks, max_blocks;
  int log2_urows;    // rows per K/V copy: min(block_size, 64)
  int tiles;         // query tiles per (sequence, kv head) at the longest chunk (max_q_len)
  int tile_block;    // min(kTileBlock, tiles)
  int pairs;         // num_seqs * num_kv_heads
  int total;         // pairs * tiles rounded up to whole blocks
  float scale_log2;  // scale * k_scale * log2(e)
  float v_scale;     // E4M3 cache: stored V value x v_scale (1 otherwise)
  int out_bf16;      // queries and output are bf16 (else f16)
  unsigned long long wait_ns;  // limit of a wait on another role (1 s unless a test shortened it)
  int stall_cta;     // testing: this CTA's MMA issuer stops after its first S group (-1: none)
};

// A published work item; s < 0 ends the work.
struct PfItem {
  int s, g, t0, n, L, q0, ntiles, pad;
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

// KV: the pools' element type. An E4M3 cache is widened to f16 in shared memory (every E4M3
// value is an f16 value) and multiplied on the f16 tensor-core path; bf16 queries are moved to
// f16 with a power-of-two scale per row (undone in the score scale).
template <int D, int G, int KV>
__global__ void __launch_bounds__(kPfThreads, 2)
    pa_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const __grid_constant__ PrefillParams p) {
  constexpr bool BF16 = KV == kPfBF16;  // operand type of the MMAs (f16 for F16 and E4M3)
  constexpr bool kFp8 = KV == kPfE4M3;
  static_assert(!kFp8 || D == 128, "the E4M3 cache is built for head_dim 128");
  constexpr int kRegions = D / 64;
  constexpr int kTokens = kPfRows / G;
  constexpr uint32_t kQRegion = kPfRows * 128;        // 16 KiB
  constexpr uint32_t kKVRegion = kPfKeys * 128;       // 8 KiB
  constexpr uint32_t kKVBytes = kRegions * kKVRegion;  // K (or V) of one stage

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_q_heads;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  uint8_t* bp = smem_raw;
  if ((base & 1023u) != 0) {  // the swizzled operands need 1024-byte alignment
    if (tid == 0) flag_error(p.err, kErrTimeout);
    return;
  }
  const uint32_t sQ = base;
  const uint32_t sKV = sQ + kRegions * kQRegion;  // stage st: K at sKV + 2 st kKVBytes, V after it
  uint8_t* ctl = bp + (sKV + kPfStages * 2 * kKVBytes - base);
  // K and V stream through separate rings: K of tile j is free once S_j is computed, V once
  // PV_j is, so K loads run a whole softmax ahead of V loads. Every phase below counts tiles
  // (or items) over the whole run of the CTA. Tile j uses stage j % 2 of both rings, S buffer
  // j % 2 (whose first 32 columns then take P_j, read by PV_j from tensor memory), barriers
  // p_full[j % 2] and completion barriers s_full[j % 2] and o_done[j % 2]; with one commit per MMA
  // group (a second one per group slows the MMA stream by about a tenth), those two barriers
  // also release the stage's K and V to the producers (each producer waits on every phase of
  // its own stage, so a parity wait cannot pass on a phase that is still one behind). The query
  // loader does not see every phase of s_full, so the query buffer has its own barrier,
  // committed after an item's last S.
  static_assert(kPfStages == 2, "the completion barriers double as the rings' empty barriers");
  uint64_t* k_full = reinterpret_cast<uint64_t*>(ctl);  // [kPfStages]
  uint64_t* v_full = k_full + kPfStages;                 // [kPfStages]
  uint64_t* s_full = v_full + kPfStages;                 // [2] S_j complete: K_j free too
  uint64_t* p_full = s_full + 2;                         // [2] P_j written (4 warps)
  uint64_t* o_done = p_full + 2;                         // [2] PV_j complete: V_j and S buffer free
  uint64_t* o_free = o_done + 2;                         // O read by the epilogue (4 warps)
  uint64_t* q_full = o_free + 1;                         // the item's query tile landed
  uint64_t* q_empty = q_full + 1;                        // the item's last S complete
  uint64_t* item_full = q_empty + 1;                     // [kSlots]
  uint64_t* item_empty = item_full + kSlots;             // [kSlots]
  uint64_t* drain = item_empty + kSlots;
  PfItem* items = reinterpret_cast<PfItem*>(drain + 1);  // [kSlots]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(items + kSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // E4M3 cache only: the raw bytes of tile J land in the upper half of stage J % 2 and
  // complete on k_raw / v_raw; the producer warp then widens them into the stage and arrives on
  // k_full / v_full. q_ready[slot] completes when the query tile of the item in that slot is
  // in f16 and its rows' exponents are in q_exp[slot].
  uint64_t* k_raw = reinterpret_cast<uint64_t*>(ctl + 256);  // [kPfStages]
  uint64_t* v_raw = k_raw + kPfStages;                        // [kPfStages]
  uint64_t* q_ready = v_raw + kPfStages;                      // [kSlots]
  int8_t* q_exp = reinterpret_cast<int8_t*>(ctl + 384);       // [kSlots][kPfRows]

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(smem_addr(k_full + i), 1);
      mbar_init(smem_addr(v_full + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(s_full + i), 1);
      mbar_init(smem_addr(p_full + i), 4);
      mbar_init(smem_addr(o_done + i), 1);
    }
    mbar_init(smem_addr(o_free), 4);
    mbar_init(smem_addr(q_full), 1);
    mbar_init(smem_addr(q_empty), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(item_full + i), 1);
      mbar_init(smem_addr(item_empty + i), kItemReaders);
    }
    mbar_init(smem_addr(drain), 1);
    if constexpr (kFp8) {
      for (int i = 0; i < kPfStages; ++i) {
        mbar_init(smem_addr(k_raw + i), 1);
        mbar_init(smem_addr(v_raw + i), 1);
      }
      for (int i = 0; i < kSlots; ++i) mbar_init(smem_addr(q_ready + i), 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem, tS = tmem + 128;
  auto fail = [&]() {
    flag_error(p.err, kErrTimeout);
    *abort_flag = 1;
  };

  if (warp == 3) {
    // ------------------------------------------------------------------ items and queries
    // Lane 0 takes the items and loads their query tiles. With an E4M3 cache the whole warp
    // then widens each landed tile to f16 (rows lane, lane + 32, ... : one row per lane at a
    // time) and publishes it on q_ready[slot].
    if (kFp8 || lane == 0) {
      const uint64_t qpol = policy_evict_first();  // each query tile is read once
      if (lane == 0) prefetch_tensormap(&qmap);
      int k = 0, fetched = 0;
      for (;;) {
        PfItem it{-1, 0, 0, 0, 0, 0, 0, 0};
        const int slot = k % kSlots;
        bool loaded = false;
        if (lane == 0) {
          while (!*abort_flag) {
            const int v = p.work != nullptr
                              ? atomicAdd(p.work, 1)
                              : static_cast<int>(blockIdx.x) + fetched * static_cast<int>(gridDim.x);
            ++fetched;
            if (v >= p.total) break;
            const int per_block = p.pairs * p.tile_block;
            const int blk = v / per_block, rem = v - blk * per_block;
            const int sg = rem / p.tile_block;
            const int tile = p.tiles - 1 - (blk * p.tile_block + (rem - sg * p.tile_block));
            if (tile < 0) continue;  // past the shortest tile (the last block is partial)
            const int s = sg / p.num_kv_heads, g = sg - s * p.num_kv_heads;
            const int q0 = __ldg(p.q_starts + s);
            const int n = __ldg(p.q_starts + s + 1) - q0;
            const int t0 = tile * kTokens;
            if (t0 >= n) continue;  // the chunk is shorter than this tile
            const int L = __ldg(p.ctx_lens + s);
            const bool rows_ok = q0 >= 0 && q0 + n <= p.num_tokens;
            // invalid lengths (or a chunk longer than max_q_len): the tile's rows are zero
            if (!rows_ok || n > L || L > p.max_blocks * p.block_size || n > p.tiles * kTokens) {
              flag_error(p.err, kErrCtxLen);
              if (rows_ok) {
                const int tend = min(n, t0 + kTokens);
                for (int t = t0; t < tend; ++t)
                  for (int i = 0; i < G * D / 8; ++i)
                    reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                             (static_cast<size_t>(q0 + t) * Hq + g * G) * D)[i] =
                        make_uint4(0, 0, 0, 0);
              }
              continue;
            }
            // causal extent of the tile: its last query stands at position L - n + t_last
            const int t_last = min(n, t0 + kTokens) - 1;
            it = PfItem{s, g, t0, n, L, q0, (L - n + t_last + 1 + kPfKeys - 1) / kPfKeys, 0};
            break;
          }
          if (k >= kSlots &&
              !mbar_wait_bounded(smem_addr(item_empty + slot), ((k / kSlots) - 1) & 1, p.wait_ns)) {
            fail();
            it.s = -1;
          }
          items[slot] = it;
          mbar_arrive(smem_addr(item_full + slot));
          // the query buffer is free once the previous item's last S MMA has completed
          if (it.s >= 0 &&
              (k == 0 || mbar_wait_bounded(smem_addr(q_empty), (k - 1) & 1, p.wait_ns))) {
            mbar_arrive_expect_tx(smem_addr(q_full), kRegions * kQRegion);
#pragma unroll
            for (int c = 0; c < kRegions; ++c)
              tma_load_3d(sQ + c * kQRegion, &qmap, c * 64, it.g * G, it.q0 + it.t0,
                          smem_addr(q_full), qpol);
            loaded = true;
          } else if (it.s >= 0) {
            fail();
          }
        }
        if constexpr (kFp8) loaded = __shfl_sync(0xffffffffu, loaded, 0);
        if (!loaded) break;
        const int kq = k++;
        if constexpr (kFp8) {
          const bool landed =
              __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(q_full), kq & 1, p.wait_ns));
          if (!landed) {
            if (lane == 0) fail();
            break;
          }
          // bf16 queries: row r times 2^e_r, with e_r putting the row's largest magnitude in
          // [2^14, 2^15), is exact in f16 for every element above f16's subnormal range
          for (int r = lane; r < kPfRows; r += 32) {
            int e = 0;
            if (p.out_bf16) {
              float amax = 0.f;
#pragma unroll
              for (int c = 0; c < 8 * kRegions; ++c) {
                const uint4 v = lds128(sQ + (c / 8) * kQRegion + sw128_offset(r, c % 8));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f = bf16x2_to_float2(w[i]);
                  amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
              }
              if (amax > 0.f && amax < INFINITY) e = max(-120, min(120, 14 - ilogbf(amax)));
              const float up = ldexpf(1.f, e);
#pragma unroll
              for (int c = 0; c < 8 * kRegions; ++c) {
                const uint32_t a = sQ + (c / 8) * kQRegion + sw128_offset(r, c % 8);
                const uint4 v = lds128(a);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f = bf16x2_to_float2(w[i]);
                  h[i] = pack16<false>(f.x * up, f.y * up);
                }
                *reinterpret_cast<uint4*>(bp + (a - base)) = make_uint4(h[0], h[1], h[2], h[3]);
              }
            }
            q_exp[slot * kPfRows + r] = static_cast<int8_t>(e);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(q_ready + slot));
        }
      }
      // no query copy may still be landing when the CTA exits (matters after an abort)
      if (lane == 0 && k >= 1) mbar_wait_bounded(smem_addr(q_full), (k - 1) & 1, kDrainLimitNs);
    }
  } else if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ K/V producers
    // warp 0 streams K, warp 2 streams V, each through its own ring (two lanes of one warp
    // would hold each other up in their barrier waits). Lane 0 issues the copies. With an E4M3
    // cache the copies bring the raw bytes into the upper half of the stage and the whole warp
    // then widens them to f16 in place (a raw row sits where its f16 upper half goes, so each
    // row is read by its lanes before any of them writes).
    if (kFp8 || lane == 0) {
      // the warp's decisions must be uniform when all its lanes take part
      auto all = [](bool v) -> bool {
        if constexpr (kFp8) return __all_sync(0xffffffffu, v) != 0;
        return v;
      };
      auto any = [](bool v) -> bool {
        if constexpr (kFp8) return __any_sync(0xffffffffu, v) != 0;
        return v;
      };
      const bool is_v = warp == 2;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      uint64_t* fullb = is_v ? v_full : k_full;
      uint64_t* rawb = is_v ? v_raw : k_raw;      // E4M3: raw copies landed
      uint64_t* copyb = kFp8 ? rawb : fullb;      // the barrier the copies complete on
      uint64_t* emptyb = is_v ? o_done : s_full;  // stage st of tile J - 2 consumed
      const uint64_t pol = policy_evict_normal();  // the sequence's other query tiles reread them
      const int urows = 1 << p.log2_urows, B = p.block_size;
      const int units = kPfKeys >> p.log2_urows;
      // bytes of one copy unit, and where a tile's copies land within the stage
      constexpr uint32_t kUnitRowBytes = kFp8 ? 128u : static_cast<uint32_t>(kRegions) * 128u;
      constexpr uint32_t kLandOffset = kFp8 ? kKVRegion : 0u;
      if (lane == 0) prefetch_tensormap(map);
      int J = 0;  // tiles issued, over all items
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k % kSlots;
        if (!all(mbar_wait_bounded(smem_addr(item_full + slot), (k / kSlots) & 1, p.wait_ns))) {
          if (lane == 0) fail();
          break;
        }
        const PfItem it = items[slot];
        if (any(it.s < 0 || *abort_flag)) break;
        const int32_t* trow = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks;
        // The block-table entries of tile j + 1 are read while the producer waits for a free
        // stage for tile j + 1, so their latency is off the copy path.
        int ph[8];
        auto load_phys = [&](int j) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int key = j * kPfKeys + u * urows;
            ph[u] = (u < units && key < it.L) ? __ldg(trow + (key >> p.log2_block)) : -2;
          }
        };
        load_phys(0);
        for (int j = 0; j < it.ntiles; ++j, ++J) {
          const int st = J % kPfStages;
          if (J >= kPfStages &&
              !all(mbar_wait_bounded(smem_addr(emptyb + st), ((J / kPfStages) - 1) & 1,
                                     p.wait_ns))) {
            if (lane == 0) fail();
            ok = false;
            break;
          }
          if (any(*abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sKV + 2 * st * kKVBytes + (is_v ? kKVBytes : 0u);
          if (lane == 0) {
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
                rowc[u] = (ph[u] * p.num_kv_heads + it.g) * B + (key & (B - 1));
                bytes += kUnitRowBytes * static_cast<uint32_t>(urows);
              }
            }
            const uint32_t bar = smem_addr(copyb + st);
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (rowc[u] < 0) continue;
              if constexpr (kFp8) {
                tma_load_2d(dst + kLandOffset + static_cast<uint32_t>(u * urows * 128), map, 0,
                            rowc[u], bar, pol);
              } else {
#pragma unroll
                for (int c = 0; c < kRegions; ++c)
                  tma_load_2d(dst + c * kKVRegion + static_cast<uint32_t>(u * urows * 128), map,
                              c * 64, rowc[u], bar, pol);
              }
            }
          }
          if constexpr (kFp8) {
            // widen the tile: lane (row r % 4 of a group of 4 rows, 16-byte chunk c) turns 16
            // E4M3 values into two 16-byte f16 chunks of the row's region c / 4
            if (!all(mbar_wait_bounded(smem_addr(rawb + st), (J / kPfStages) & 1, p.wait_ns))) {
              if (lane == 0) fail();
              ok = false;
              ++J;  // its copies were issued: the drain below waits for them
              break;
            }
            const int rr = lane >> 3, c = lane & 7;
            uint8_t* stage = bp + (dst - base);
#pragma unroll 4
            for (int r0 = 0; r0 < kPfKeys; r0 += 4) {
              const int r = r0 + rr;
              const uint4 v =
                  *reinterpret_cast<const uint4*>(stage + kLandOffset + sw128_offset(r, c));
              __syncwarp();
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
              uint32_t h[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                h[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xffffu));
                h[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
              }
              uint8_t* region = stage + (c >> 2) * kKVRegion;
              const int c0 = 2 * (c & 3);
              *reinterpret_cast<uint4*>(region + sw128_offset(r, c0)) =
                  make_uint4(h[0], h[1], h[2], h[3]);
              *reinterpret_cast<uint4*>(region + sw128_offset(r, c0 + 1)) =
                  make_uint4(h[4], h[5], h[6], h[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(fullb + st));
          }
          if (j + 1 < it.ntiles) load_phys(j + 1);
        }
        if (ok && lane == 0) mbar_arrive(smem_addr(item_empty + slot));
      }
      // no copy of this CTA may still be landing when it exits (matters after an abort)
      if (lane == 0)
        for (int jj = max(0, J - kPfStages); jj < J; ++jj)
          mbar_wait_bounded(smem_addr(copyb + jj % kPfStages), (jj / kPfStages) & 1,
                            kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_f16(kPfRows, kPfKeys, BF16, false);
      // Shared-memory descriptors are built once: an operand at byte offset o from a base has
      // the base's descriptor plus o / 16 in the start-address field (no carry: every address
      // is below 256 KB). The tensor pipe cannot run ahead of this thread, so every instruction
      // between two MMAs lengthens the MMA stream; with the descriptors rebuilt per MMA the
      // attention sequence ran at half the pipe's rate.
      const uint64_t dQ = umma_sdesc(sQ, 16, 1024);
      const uint64_t dK = umma_sdesc(sKV, 16, 1024);
      const uint64_t dV = umma_sdesc(sKV + kKVBytes, kKVRegion, 1024);
      constexpr uint32_t idO = umma_idesc_f16(kPfRows, D, BF16, true);
      // Two cursors over the items: S_ns is issued as soon as K_ns has landed (and its S buffer
      // is free, and at an item's first tile its queries have landed), PV_npv as soon as P_npv
      // and V_npv are ready (and, at an item's first tile, once the epilogue has read O),
      // whichever comes first, PV before S when both are. S runs ahead of PV by up to two
      // tiles, across item boundaries. S buffer b is free once the PV that read P from it two
      // tiles earlier has completed: tcgen05 orders MMAs of one thread only when they share an
      // accumulator, so issuing S after that PV would not be enough.
      int kS = 0, jS = 0, ns = 0;   // S stream: item, tile in item, S issued over all items
      bool haveS = false, endS = false;
      PfItem iS{};
      int kP = 0, jP = 0, npv = 0;  // PV stream: item, tile in item, PV issued over all items
      bool haveP = false;
      PfItem iP{};
      int nO = 0;  // items whose O is complete
      bool ok = true;
      const bool stalled = static_cast<int>(blockIdx.x) == p.stall_cta;
      uint32_t idle = 0;
      unsigned long long idle_since = 0;
      for (;;) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        bool did = false;
        // ---- PV stream (first: PV_j stands between P_j and the softmax's write of P_{j+1},
        // while S runs up to two tiles ahead)
        if (!haveP) {
          if (kP < kS || (kP == kS && haveS)) {
            iP = items[kP % kSlots];
            haveP = true;
            jP = 0;
          } else if (endS && kP == kS) {
            break;  // every item is done
          }
        }
        if (haveP && npv < ns && !stalled) {
          const int stp = npv % kPfStages;
          if (mbar_test(smem_addr(p_full + stp), (npv >> 1) & 1) &&
              mbar_test(smem_addr(v_full + stp), (npv / kPfStages) & 1) &&
              (jP > 0 || nO == 0 || mbar_test(smem_addr(o_free), (nO - 1) & 1))) {
            tc_fence_after();
            const uint64_t dVs = dV + ((2u * stp * kKVBytes) >> 4);
            const uint32_t tP = tS + 64 * stp;
#pragma unroll
            for (int k = 0; k < kPfKeys / 16; ++k)
              umma_f16_ta(tO, tP + 8 * k, dVs + k * 128, idO, jP > 0 || k > 0);
            umma_commit(smem_addr(o_done + stp));
            ++npv;
            if (++jP == iP.ntiles) {
              ++nO;
              mbar_arrive(smem_addr(item_empty + kP % kSlots));
              haveP = false;
              ++kP;
            }
            did = true;
          }
        }
        // ---- S stream
        if (!haveS && !endS && mbar_test(smem_addr(item_full + kS % kSlots), (kS / kSlots) & 1)) {
          iS = items[kS % kSlots];
          if (iS.s < 0) {
            endS = true;
          } else {
            haveS = true;
            jS = 0;
          }
          did = true;
        }
        if (haveS && !(stalled && ns >= 1)) {
          const int st = ns % kPfStages, b = ns & 1;
          if (mbar_test(smem_addr(k_full + st), (ns / kPfStages) & 1) &&
              (ns < 2 || mbar_test(smem_addr(o_done + b), ((ns >> 1) - 1) & 1)) &&
              (jS > 0 || (kFp8 ? mbar_test(smem_addr(q_ready + kS % kSlots), (kS / kSlots) & 1)
                                : mbar_test(smem_addr(q_full), kS & 1)))) {
            tc_fence_after();
            const uint64_t dKs = dK + ((2u * st * kKVBytes) >> 4);
            const uint32_t dS = tS + 64 * b;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              constexpr uint32_t kQStep = kQRegion >> 4, kKStep = kKVRegion >> 4;
              const uint32_t c = k / 4, kk = k % 4;
              umma_f16(dS, dQ + (c * kQStep + kk * 2), dKs + (c * kKStep + kk * 2), idS, k > 0);
            }
            umma_commit(smem_addr(s_full + b));
            ++ns;
            if (++jS == iS.ntiles) {
              umma_commit(smem_addr(q_empty));
              haveS = false;
              ++kS;
            }
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (idle++ == 0) {
          idle_since = global_ns();
        } else if ((idle & 63u) == 0 && global_ns() - idle_since > p.wait_ns) {
          ok = false;
          break;
        }
      }
      if (!ok) fail();
      // every MMA this thread issued has completed before tensor memory is released
      umma_commit(smem_addr(drain));
      mbar_wait_bounded(smem_addr(drain), 0, kDrainLimitNs);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------------ softmax warpgroup
    const int r = tid - kSoftmaxWarp0 * 32;  // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp - kSoftmaxWarp0) * 32) << 16;
    int jx = 0;  // tiles processed, over all items
    bool ok = true;
    // An item's epilogue (O / l to its rows, then O and the item slot released) is deferred
    // into the next item's first tile, after that tile's weights are computed and its P is
    // written: the wait for the item's last PV (PV_{j-1} of that tile, waited for just before)
    // then overlaps useful work.
    bool pend = false, pend_valid = false;
    float pend_inv = 0.f;
    uint4* pend_dst = nullptr;
    int pend_slot = 0;
    // output rows in the query dtype: the MMA operand type, except for an E4M3 cache (f16
    // operands, bf16 or f16 output)
    auto pack_out = [&](float lo, float hi) -> uint32_t {
      if constexpr (kFp8) return p.out_bf16 ? pack16<true>(lo, hi) : pack16<false>(lo, hi);
      return pack16<BF16>(lo, hi);
    };
    auto epilogue = [&]() {
      // two 32-column loads per wait: each tensor-memory round trip is on the item's path
#pragma unroll 1
      for (int c = 0; c < D; c += 64) {
        uint32_t v[2][32];
        tmem_ld32_nowait(tO + lane_base + c, v[0]);
        tmem_ld32_nowait(tO + lane_base + c + 32, v[1]);
        tmem_wait_ld();
        if (pend_valid) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_out(__uint_as_float(v[h][2 * i]) * pend_inv,
                              __uint_as_float(v[h][2 * i + 1]) * pend_inv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              pend_dst[(c + 32 * h) / 8 + i] =
                  make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(o_free));
        mbar_arrive(smem_addr(item_empty + pend_slot));
      }
      pend = false;
    };
    for (int k = 0;; ++k) {
      const int slot = k % kSlots;
      ok = mbar_wait_bounded(smem_addr(item_full + slot), (k / kSlots) & 1, p.wait_ns);
      if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
        ok = false;
        break;
      }
      const PfItem it = items[slot];
      if (it.s < 0) break;
      // scores are scaled into the log2 domain by scale * k_scale * log2(e), and, for queries
      // widened from bf16, by the row's 2^-e as well
      float row_scale = p.scale_log2;
      if constexpr (kFp8) {
        ok = mbar_wait_bounded(smem_addr(q_ready + slot), (k / kSlots) & 1, p.wait_ns);
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        row_scale = ldexpf(p.scale_log2, -static_cast<int>(q_exp[slot * kPfRows + r]));
      }
      const int tr = it.t0 + r / G;
      const bool row_valid = tr < it.n;
      const int pos = it.L - it.n + tr;  // last position this row may see
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.ntiles; ++j, ++jx) {
        const int b = jx & 1;
        ok = mbar_wait_bounded(smem_addr(s_full + b), (jx >> 1) & 1, p.wait_ns);
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
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

        const int key0 = j * kPfKeys;
        // Rows that see all 64 keys of the tile (every tile before the diagonal) need no mask.
        // Scores stay raw until the exponent: m is kept in scaled log2 units and the weight of
        // score x is 2^(x * scale_log2 - m), one FFMA and one ex2.
        const bool full = row_valid && key0 + kPfKeys - 1 <= pos;
        const int lim = row_valid ? pos - key0 : -1;  // last visible column (full: >= 63)
        float mt = -INFINITY;
        if (full) {
          // four independent chains of 3-input maxima over 16 scores each
          float a[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float* y = x + 16 * q;
            float t = fmax3(y[0], y[1], y[2]);
#pragma unroll
            for (int i = 3; i < 15; i += 2) t = fmax3(t, y[i], y[i + 1]);
            a[q] = fmaxf(t, y[15]);
          }
          mt = fmax3(a[0], a[1], fmaxf(a[2], a[3]));
        } else {
#pragma unroll
          for (int c = 0; c < kPfKeys; ++c)
            if (c <= lim) mt = fmaxf(mt, x[c]);
        }
        mt = mt == -INFINITY ? -INFINITY : mt * row_scale;
        // Lazy rescaling: the row keeps its reference maximum m unless the tile's maximum
        // exceeds it by more than 8 (log2 units); weights then stay below 2^8 and O is rescaled
        // rarely. Numerator and denominator share the same reference, so the result is
        // unchanged.
        const float m_new = mt > m + 8.f ? mt : m;
        const float alpha = m_new == m ? 1.f : ex2(m - m_new);
        uint32_t pk[kPfKeys / 2];
        float psum = 0.f;
        if (full) {
          // pairs of scores through one packed FMA; the row sum in two packed partial sums
          const uint64_t sc2 = f2pack(row_scale, row_scale), nm2 = f2pack(-m_new, -m_new);
          uint64_t s2 = f2pack(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kPfKeys; c += 2) {
            float t0, t1;
            f2unpack(ffma2(f2pack(x[c], x[c + 1]), sc2, nm2), t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            pk[c / 2] = pack16<BF16>(p0, p1);
            s2 = fadd2(s2, f2pack(p0, p1));
          }
          float s0, s1;
          f2unpack(s2, s0, s1);
          psum = s0 + s1;
        } else {
#pragma unroll
          for (int c = 0; c < kPfKeys; c += 2) {
            const float p0 =
                c <= lim && m_new != -INFINITY ? ex2(fmaf(x[c], row_scale, -m_new)) : 0.f;
            const float p1 = c + 1 <= lim && m_new != -INFINITY
                                 ? ex2(fmaf(x[c + 1], row_scale, -m_new))
                                 : 0.f;
            pk[c / 2] = pack16<BF16>(p0, p1);
            psum += p0 + p1;
          }
        }
        l = l * alpha + psum;
        m = m_new;

        // P_j goes to its own S buffer, so only reading or rescaling O waits for PV_{j-1}: the
        // previous item's epilogue (at an item's first tile) and a rescale (rare)
        const bool rescale = j >= 1 && __any_sync(0xffffffffu, alpha != 1.f);
        const bool epi = j == 0 && pend;
        if (rescale || epi) {
          ok = mbar_wait_bounded(smem_addr(o_done + ((jx - 1) & 1)), ((jx - 1) >> 1) & 1, p.wait_ns);
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        bool zeroed = false;
        if (j == it.ntiles - 1 && key0 + kPfKeys > it.L) {
          // value rows past the cache's last position (stale slots, or not loaded) become zero,
          // so that zero weights cannot meet a NaN; the tile's V copies must have landed first
          ok = mbar_wait_bounded(smem_addr(v_full + (jx % kPfStages)), (jx / kPfStages) & 1,
                                 p.wait_ns);
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
          const uint32_t vst = sKV + 2 * (jx % kPfStages) * kKVBytes + kKVBytes;
          const int r0 = it.L - key0;
          const int nbytes16 = (kPfKeys - r0) * 8 * kRegions;  // 16-byte chunks to clear
          for (int i = r; i < nbytes16; i += 128) {
            const int c = i % (8 * kRegions), row = r0 + i / (8 * kRegions);
            *reinterpret_cast<uint4*>(bp + (vst - base) + (c / 8) * kKVRegion + row * 128 +
                                      (c % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          zeroed = true;
        }
        // P row r into the first 32 columns of S buffer b (S_j has been read)
        tmem_st32_nowait(tS + 64 * b + lane_base, pk);
        if (epi) epilogue();  // the previous item's O is complete (waited above)
        if (rescale) {
#pragma unroll 1
          for (int c = 0; c < D; c += 16) {
            float v[16];
            tmem_ld16(tO + lane_base + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha;
            tmem_st16(tO + lane_base + c, v);
          }
        }
        tmem_wait_st();
        if (zeroed) fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(p_full + b));
      }
      if (!ok) break;
      // ---- the item's epilogue is deferred (see above)
      pend = true;
      pend_valid = row_valid;
      if constexpr (kFp8)
        pend_inv = l > 0.f ? p.v_scale / l : 0.f;
      else
        pend_inv = l > 0.f ? 1.f / l : 0.f;
      pend_dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                          (static_cast<size_t>(it.q0 + tr) * Hq + it.g * G + r % G) * D);
      pend_slot = slot;
    }
    if (ok && pend) {  // the last item's epilogue, once its last PV has completed
      ok = mbar_wait_bounded(smem_addr(o_done + ((jx - 1) & 1)), ((jx - 1) >> 1) & 1, p.wait_ns);
      if (__any_sync(0xffffffffu, !ok)) ok = false;
      if (ok) {
        tc_fence_after();
        epilogue();
      }
    }
    if (!ok && lane == 0) fail();
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

template <int D, int G, int KV>
cudaError_t launch_prefill(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                           const PrefillParams& p, unsigned grid, size_t smem, cudaStream_t stream) {
  auto fn = pa_prefill_kernel<D, G, KV>;
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
  fn<<<grid, kPfThreads, smem, stream>>>(qm, km, vm, p);
  return cudaGetLastError();
}

template <int D, int KV>
cudaError_t launch_prefill_g(int group, const CUtensorMap& qm, const CUtensorMap& km,
                             const CUtensorMap& vm, const PrefillParams& p, unsigned grid,
                             size_t smem, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefill<D, 1, KV>(qm, km, vm, p, grid, smem, stream);
    case 2: return launch_prefill<D, 2, KV>(qm, km, vm, p, grid, smem, stream);
    case 4: return launch_prefill<D, 4, KV>(qm, km, vm, p, grid, smem, stream);
    case 8: return launch_prefill<D, 8, KV>(qm, km, vm, p, grid, smem, stream);
    default: return launch_prefill<D, 16, KV>(qm, km, vm, p, grid, smem, stream);
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
    msg = "pa_prefill supports PA_F16 and PA_BF16 queries";
    return PA_EUNSUPPORTED;
  }
  const bool fp8 = a.kv_dtype == PA_FP8_E4M3;
  if (!fp8 && a.kv_dtype != a.dtype) {
    msg = "kv_dtype must equal dtype, or be PA_FP8_E4M3";
    return PA_EINVAL;
  }
  if (a.head_dim != 64 && a.head_dim != 128) {
    msg = "head_dim must be 64 or 128";
    return PA_EUNSUPPORTED;
  }
  if (fp8 && a.head_dim != 128) {
    msg = "an E4M3 cache is built for head_dim 128";
    return PA_EUNSUPPORTED;
  }
  if (fp8 && (!(a.k_scale > 0.f) || !(a.v_scale > 0.f) || !std::isfinite(a.k_scale) ||
              !std::isfinite(a.v_scale))) {
    msg = "k_scale and v_scale must be finite and > 0 for an E4M3 cache";
    return PA_EINVAL;
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
  const int tokens_per_tile = kPfRows / group;
  const long long tiles = (a.max_q_len + tokens_per_tile - 1) / tokens_per_tile;
  const long long tile_block = std::min<long long>(kTileBlock, tiles);
  const long long total = (tiles + tile_block - 1) / tile_block * tile_block *
                          static_cast<long long>(a.num_seqs) * a.num_kv_heads;
  if (total >= (1ll << 30)) {
    msg = "more than 2^30 work items (sequences x kv heads x query tiles)";
    return PA_EUNSUPPORTED;
  }
  const int urows = std::min(a.block_size, kPfKeys);
  CUtensorMap qmap, kmap, vmap;
  pa_status st = encode_query_tile_map(&qmap, a.q, a.num_tokens, a.num_q_heads, a.head_dim, group,
                                       tokens_per_tile, msg);
  if (st != PA_OK) return st;
  const int elt = fp8 ? 1 : 2;
  st = encode_pool_rows_map(&kmap, a.k_pool, rows, a.head_dim, elt, urows, msg);
  if (st != PA_OK) return st;
  st = encode_pool_rows_map(&vmap, a.v_pool, rows, a.head_dim, elt, urows, msg);
  if (st != PA_OK) return st;

  PrefillParams p{};
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.ctx_lens = a.ctx_lens;
  p.q_starts = a.q_starts;
  p.err = a.err_flag;
  p.work = a.work_counter;
  p.num_tokens = a.num_tokens;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.log2_block = 0;
  while ((1 << p.log2_block) < a.block_size) ++p.log2_block;
  p.log2_urows = 0;
  while ((1 << p.log2_urows) < urows) ++p.log2_urows;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks_per_seq;
  p.tiles = static_cast<int>(tiles);
  p.tile_block = static_cast<int>(tile_block);
  p.pairs = a.num_seqs * a.num_kv_heads;
  p.total = static_cast<int>(total);
  p.scale_log2 = a.scale * (fp8 ? a.k_scale : 1.f) * 1.4426950408889634f;
  p.v_scale = fp8 ? a.v_scale : 1.f;
  p.out_bf16 = a.dtype == PA_BF16 ? 1 : 0;
  p.wait_ns = launch_wait_ns();
  p.stall_cta = launch_stall_cta();

  const int D = a.head_dim;
  const size_t regions = static_cast<size_t>(D / 64);
  // no alignment slack: the kernel needs (and checks) a 1024-byte aligned dynamic region, and
  // two CTAs then fit on an SM
  const size_t smem = regions * kPfRows * 128 + kPfStages * 2 * regions * kPfKeys * 128 +
                      (fp8 ? kCtlBytesFp8 : kCtlBytes);
  const int sms = device_sm_count();
  if (sms <= 0) {
    msg = "cannot read the SM count of the current device";
    return PA_ECUDA;
  }
  const unsigned grid = static_cast<unsigned>(std::min<long long>(2ll * sms, total));
  if (a.work_counter != nullptr) {
    st = cuda_status(cudaMemsetAsync(a.work_counter, 0, sizeof(int32_t), stream),
                     "pa_prefill work counter reset", msg);
    if (st != PA_OK) return st;
  }
  const bool bf16 = a.dtype == PA_BF16;
  cudaError_t e;
  if (fp8)
    e = launch_prefill_g<128, kPfE4M3>(group, qmap, kmap, vmap, p, grid, smem, stream);
  else if (D == 128)
    e = bf16 ? launch_prefill_g<128, kPfBF16>(group, qmap, kmap, vmap, p, grid, smem, stream)
             : launch_prefill_g<128, kPfF16>(group, qmap, kmap, vmap, p, grid, smem, stream);
  else
    e = bf16 ? launch_prefill_g<64, kPfBF16>(group, qmap, kmap, vmap, p, grid, smem, stream)
             : launch_prefill_g<64, kPfF16>(group, qmap, kmap, vmap, p, grid, smem, stream);
  return cuda_status(e, "pa_prefill kernel launch", msg);
}

}  // namespace pa
