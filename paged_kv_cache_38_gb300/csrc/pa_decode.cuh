// pa_decode.cuh - paged decode attention kernels for sm_103a (templates; instantiated per KV dtype).
//
// Method: "Efficient Memory Management for Large Language Model Serving with PagedAttention"
// (paper summary page), paragraph on the PagedAttention kernel: the keys of logical block j sit
// in a physical block found through the sequence's block table; the kernel fetches every block
// wherever it is stored, scores the query against it and combines the values, and the result
// equals ordinary attention. "Continuous Batching and PagedAttention", section "The block table
// is a page table": the kernel gathers through the table instead of striding.
//
// GB300 design: a persistent kernel, one CTA of 13 warps per SM.
//   * Work items are (sequence, kv head, context split) in sequence order; CTAs take the next
//     item from a global counter, so the items of sequences that share prompt blocks run at the
//     same time on different SMs and the shared blocks are served from L2.
//   * Warp 0 schedules: it keeps up to 2 items queued in shared memory -- descriptor, the
//     item's block-table slice (one coalesced load, out-of-pool ids masked and flagged) and the
//     group's queries (one bulk copy).
//   * Warps 1..4 produce: tile g of the CTA's tile sequence is issued by warp 1 + g % 4 as 2-D
//     TMA tensor copies of each (block, kv head) tile of K and V into a ring of shared-memory
//     stages (128-byte swizzle) completing on mbarriers. Several issuing warps are needed: one
//     warp's in-order stream of copies reaches only a fraction of an SM's share of HBM
//     bandwidth. The ring runs across item boundaries, so HBM traffic does not stop between items.
//   * Warps 5..12 consume: tile t of an item goes to consumer t % 8, each keeping its own
//     online-softmax state (running max in log2 units, running sum, fp32 accumulator).
//     Group size G <= 2: warp-shuffle dot products on the CUDA cores. G >= 4: the GQA group makes
//     each 16-token tile a small dense contraction, done with mma.sync m16n8k16
//     (S^T = K Q^T with the G query heads as the N dimension, then O^T += V^T P^T).
//   * At the end of an item the consumer states are merged in shared memory; an item that covers
//     its sequence's whole context writes the output, otherwise fp32 partials (split-K, flash-
//     decoding style). When every CTA has run out of items, one grid-wide barrier (cooperative
//     launch) separates the item phase from the combine phase, in which every warp of the grid
//     combines the partials of one (sequence, query head). (Publishing each split with its own
//     GPU-scope fence was measured slower: it stalls the consumers at every item.)
#pragma once

#include <mutex>
#include <set>
#include <utility>

#include "pa_device.cuh"

namespace pa {

enum KvKind { kKvF16 = 0, kKvBF16 = 1, kKvE4M3 = 2 };

constexpr int kProducerWarps = 4;
constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = 32 * (1 + kProducerWarps + kConsumerWarps);
constexpr int kMaxStages = 32;
constexpr int kItemSlots = 2;          // work items queued ahead by the scheduler warp
constexpr int kMaxItemUnits = 256;     // copy units (table rows) of one work item
constexpr int kMaxSeqsPerLaunch = 4096;
constexpr int kScanWarps = kDecodeThreads / 32;
constexpr int kRemBuckets = 32;  // size classes of the last-split items (longest first)
// ints of the prologue's scan area for n sequences: two prefix arrays, the part-2 order, the
// warp totals and the per-warp bucket counts
__host__ __device__ constexpr size_t scan_ints(size_t n) {
  return 3 * n + 2 + 2 * kScanWarps + kScanWarps * kRemBuckets + 2 * kRemBuckets;
}
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  float* part_o;        // [num_seqs][num_q_heads][max_splits][D] unnormalised, v_scale applied
  float2* part_ml;      // [num_seqs][num_q_heads][max_splits] (max score in log2 units, weight sum)
  unsigned long long* counters;  // [0] next item, [1] CTAs finished, [2] grid barrier (id-tagged)
  uint32_t launch_id;
  int32_t* err;
  int num_seqs, num_q_heads, num_kv_heads;
  int block_size, log2_block, num_blocks, max_blocks, max_ctx;
  int log2_srows;       // log2 of the rows per (block, kv head) copy: min(block_size, stage_tokens)
  int split_tokens;     // tokens per work item, a multiple of max(16, block_size)
  int max_splits;       // ceil(max_ctx / split_tokens)
  int stages;           // shared-memory ring depth, a multiple of kConsumerWarps
  int region_stride;    // bytes of one 128-byte-wide column region of one copy in a stage
  int stage_bytes;      // bytes of K (or V) in one stage
  int stage_tokens;     // tokens per stage: a multiple of 16; at most 4 blocks, or part of one
  // byte offsets from the 1024-aligned shared-memory base
  int off_merge, off_q, off_bar, off_meta, off_items, off_tbl, off_scan;
  int tbl_stride;       // block-table entries per item slot
  float score_scale;    // scale * k_scale * log2(e)
  float v_scale;
  int q_bf16;           // query / output dtype is bf16 (else f16)
  unsigned long long wait_ns;  // limit of a wait on another warp or CTA (1 s unless a test
                               // shortened it)
  int stall_cta;        // testing: this CTA withholds its grid-barrier arrival (-1: none)
};

// Work item handed from the scheduler warp to the producers and consumers in shared memory.
struct ItemDesc {
  int seq;      // -1: no more work
  int kvh;
  int split;
  int nsplit;   // splits of this sequence
  int ntiles;   // ring stages of this item
  int tok0;     // first token of the item
  int tok_end;  // one past its last token
  int nunits;   // copy units of the item: srows rows of one (block, kv head) tile each; their
                // tensor-map row coordinates (or -1 for a block outside the pool) fill the slot
};

template <int KV, int D>
struct Geom {
  static constexpr int kElt = KV == kKvE4M3 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kRegions = kRowBytes / 128;  // 128-byte column regions per token row
  static constexpr int kColsPerRegion = 128 / kElt;
};


// Byte offset inside a stage tensor of (token row r of the stage, 16-byte chunk c of the row),
// matching the TMA 128-byte swizzle (chunk index XOR row-in-8) of each 1024-aligned region.
struct StageRow {
  uint32_t base;  // offset of chunk 0 of the row (region 0), without swizzle
  uint32_t x;     // row & 7
};

__device__ __forceinline__ StageRow stage_row(int r, int log2_block, int regions, int region_stride) {
  const int blk = r >> log2_block;
  const int rr = r & ((1 << log2_block) - 1);
  StageRow s;
  s.base = static_cast<uint32_t>(blk * regions * region_stride + rr * 128);
  s.x = static_cast<uint32_t>(rr & 7);
  return s;
}

__device__ __forceinline__ uint32_t chunk_addr(uint32_t tensor, StageRow row, int c,
                                               int region_stride) {
  return tensor + row.base + static_cast<uint32_t>((c >> 3) * region_stride) +
         ((static_cast<uint32_t>(c & 7) ^ row.x) << 4);
}

// ---------------------------------------------------------------------------------------------
// Consumer state and per-tile math.

// Online-softmax state of one consumer warp for the G query heads of its KV head.
template <int KV, int D, int G, bool MMA>
struct Consumer;

// ---- SIMT path (G = 1 or 2): lanes split a token row into 16-byte chunks.
template <int KV, int D, int G>
struct Consumer<KV, D, G, false> {
  using Gm = Geom<KV, D>;
  static constexpr int kCpr = Gm::kRowBytes / 16;        // lanes per token row
  static constexpr int kGroups = 32 / kCpr;               // token rows per warp step
  static constexpr int kIters = 16 / kGroups;             // steps per 16-token tile
  static constexpr int kE = 16 / Gm::kElt;                // elements per lane chunk
  static constexpr bool kBF16 = KV == kKvBF16;

  float q[G][kE];
  float acc[G][kE];
  float m[G], l[G];
  int grp, ci;

  // qs: the group's G query rows (G x D, f16 or bf16) staged in shared memory.
  __device__ void init(const uint16_t* qs, bool qbf, int lane) {
    grp = lane / kCpr;
    ci = lane % kCpr;
    for (int h = 0; h < G; ++h) {
      const uint16_t* row = qs + h * D + ci * kE;
      for (int e = 0; e < kE; e += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + e);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        for (int k = 0; k < 4; ++k) {
          const float2 f = qbf ? bf16x2_to_float2(w[k]) : f16x2_to_float2(w[k]);
          q[h][e + 2 * k] = f.x;
          q[h][e + 2 * k + 1] = f.y;
        }
      }
      for (int e = 0; e < kE; ++e) acc[h][e] = 0.f;
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
  }

  // The lane's chunk of one token row as kE floats.
  __device__ static void load_row(uint32_t addr, float (&x)[kE]) {
    const uint4 v = lds128(addr);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (KV == kKvE4M3) {
      for (int k = 0; k < 4; ++k) {
        const float2 a = f16x2_to_float2(e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu)));
        const float2 b = f16x2_to_float2(e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16)));
        x[4 * k] = a.x;
        x[4 * k + 1] = a.y;
        x[4 * k + 2] = b.x;
        x[4 * k + 3] = b.y;
      }
    } else {
      for (int k = 0; k < 4; ++k) {
        const float2 f = x2_to_float2<kBF16>(w[k]);
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
      }
    }
  }

  // One 16-token tile: rows r0..r0+15 of the stage, `valid` = bit mask of usable tokens. A full
  // tile (every token valid, all but an item's last tile) skips the per-row validity tests.
  __device__ void tile(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0, uint32_t valid,
                       float score_scale) {
    if (valid == 0xffffu)
      tile_impl<true>(p, ks, vs, r0, valid, score_scale);
    else
      tile_impl<false>(p, ks, vs, r0, valid, score_scale);
  }

  template <bool kFull>
  __device__ __forceinline__ void tile_impl(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0,
                                            uint32_t valid, float score_scale) {
    float s[kIters][G];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int r = it * kGroups + grp;
      const StageRow row = stage_row(r0 + r, p.log2_srows, Gm::kRegions, p.region_stride);
      float k[kE];
      load_row(chunk_addr(ks, row, ci, p.region_stride), k);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) dot = fmaf(q[h][e], k[e], dot);
#pragma unroll
        for (int off = 1; off < kCpr; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        s[it][h] = (kFull || ((valid >> r) & 1u)) ? dot * score_scale : -INFINITY;
      }
    }
    float ref[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = s[0][h];
#pragma unroll
      for (int it = 1; it < kIters; ++it) mx = fmaxf(mx, s[it][h]);
#pragma unroll
      for (int off = kCpr; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[h], mx);
      ref[h] = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = ex2(m[h] - ref[h]);
      m[h] = mnew;
      l[h] *= alpha;
#pragma unroll
      for (int e = 0; e < kE; ++e) acc[h][e] *= alpha;
    }
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int r = it * kGroups + grp;
      if (!kFull && !((valid >> r) & 1u)) continue;
      const StageRow row = stage_row(r0 + r, p.log2_srows, Gm::kRegions, p.region_stride);
      float v[kE];
      load_row(chunk_addr(vs, row, ci, p.region_stride), v);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = ex2(s[it][h] - ref[h]);
        l[h] += pr;
#pragma unroll
        for (int e = 0; e < kE; ++e) acc[h][e] = fmaf(pr, v[e], acc[h][e]);
      }
    }
  }

  // Combine the lane groups and publish (m, l, acc) of every head for the CTA merge.
  __device__ void publish(float* mrg_o, float2* mrg_ml, int cw, int lane) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = kCpr; off < 32; off <<= 1) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
        for (int e = 0; e < kE; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
      }
      if (grp == 0) {
#pragma unroll
        for (int e = 0; e < kE; ++e) mrg_o[(cw * G + h) * D + ci * kE + e] = acc[h][e];
      }
      if (lane == 0) mrg_ml[cw * G + h] = make_float2(m[h], l[h]);
    }
  }
};

// ---- Tensor-core path (G = 4, 8, 16): per 16-token tile, S^T[16 x 8n] = K Q^T, P = exp2(S - m),
// O^T[D x 8n] += V^T P^T, with mma.sync m16n8k16 and fp32 accumulators.
template <int KV, int D, int G>
struct Consumer<KV, D, G, true> {
  using Gm = Geom<KV, D>;
  static constexpr int kNT = G > 8 ? 2 : 1;      // n-tiles of 8 query heads
  static constexpr int kK = D / 16;              // k-steps of QK^T and m-tiles of PV
  static constexpr bool kFp8 = KV == kKvE4M3;
  static constexpr bool kBF16 = KV == kKvBF16;   // operand type of the MMAs (E4M3 -> f16)
  static constexpr bool kSplitP = !kFp8;         // P as hi + lo parts for 16-bit values
  static_assert(!kFp8 || D == 128, "E4M3 tensor-core path is built for head_dim 128");

  uint32_t qf[kNT][kK][2];
  float o[kNT][kK][4];
  float m[kNT][2], l[kNT][2];
  float qexp;  // 2^-e of the query pre-scaling (E4M3 path), else 1
  int g, t4;

  // qs: the group's G query rows (G x D, f16 or bf16) staged in shared memory.
  __device__ void init(const uint16_t* qs, bool qbf, int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    qexp = 1.f;
    if constexpr (kFp8) {
      // Queries go to f16 for the f16 MMA. A power-of-two pre-scale 2^e puts the largest |q|
      // of the group in [2^14, 2^15): exact for every bf16 value in f16's normal range.
      float amax = 0.f;
      for (int i = lane; i < G * D; i += 32) {
        const uint16_t b = qs[i];
        const float v = qbf ? __uint_as_float(static_cast<uint32_t>(b) << 16)
                            : __half2float(*reinterpret_cast<const __half*>(&b));
        amax = fmaxf(amax, fabsf(v));
      }
      for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      int e = 0;
      if (amax > 0.f && amax < INFINITY) e = 14 - ilogbf(amax);
      const float up = ldexpf(1.f, e);
      qexp = ldexpf(1.f, -e);
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        for (int j = 0; j < kK; ++j) {
          for (int r = 0; r < 2; ++r) {
            // logical k = 2*t4 + 8*r + {0,1} of k-step j <-> d = 32*t4 + 4*j + 2*r + {0,1}
            const int d = 32 * t4 + 4 * j + 2 * r;
            float x = 0.f, y = 0.f;
            if (n < G) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(qs + n * D + d);
              const float2 f = qbf ? bf16x2_to_float2(w) : f16x2_to_float2(w);
              x = f.x * up;
              y = f.y * up;
            }
            qf[nt][j][r] = pack2<false>(x, y);
          }
        }
      }
    } else {
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        for (int j = 0; j < kK; ++j) {
          for (int r = 0; r < 2; ++r) {
            const int d = 16 * j + 8 * r + 2 * t4;
            qf[nt][j][r] = n < G ? *reinterpret_cast<const uint32_t*>(qs + n * D + d) : 0u;
          }
        }
      }
    }
    for (int nt = 0; nt < kNT; ++nt) {
      for (int hh = 0; hh < 2; ++hh) {
        m[nt][hh] = -INFINITY;
        l[nt][hh] = 0.f;
      }
      for (int j = 0; j < kK; ++j)
        for (int c = 0; c < 4; ++c) o[nt][j][c] = 0.f;
    }
  }

  // A full tile (every token valid, all but an item's last tile) skips the validity selects and
  // masks: on the E4M3 path they were a tenth of the integer-pipe work.
  __device__ void tile(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0, uint32_t valid,
                       float score_scale) {
    if (valid == 0xffffu)
      tile_impl<true>(p, ks, vs, r0, valid, score_scale);
    else
      tile_impl<false>(p, ks, vs, r0, valid, score_scale);
  }

  template <bool kFull>
  __device__ __forceinline__ void tile_impl(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0,
                                            uint32_t valid,
                       float score_scale) {
    const int lane = (t4 | (g << 2));
    float s[kNT][4];
    for (int nt = 0; nt < kNT; ++nt)
      for (int c = 0; c < 4; ++c) s[nt][c] = 0.f;

    // ---- S^T = K Q^T
    if constexpr (kFp8) {
      // lane reads bytes [32*t4, 32*t4+32) of token rows g and g+8 (16-byte chunks 2t4, 2t4+1)
      uint32_t ka[2][16];
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const StageRow row = stage_row(r0 + g + 8 * hi, p.log2_srows, Gm::kRegions, p.region_stride);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint4 v = lds128(chunk_addr(ks, row, 2 * t4 + cc, p.region_stride));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ka[hi][cc * 8 + 2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu));
            ka[hi][cc * 8 + 2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kK; ++j) {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          mma_16816<false>(s[nt], ka[0][2 * j], ka[1][2 * j], ka[0][2 * j + 1], ka[1][2 * j + 1],
                           qf[nt][j][0], qf[nt][j][1]);
      }
    } else {
      const int i = lane >> 3;
      const StageRow row =
          stage_row(r0 + (lane & 7) + 8 * (i & 1), p.log2_srows, Gm::kRegions, p.region_stride);
#pragma unroll
      for (int j = 0; j < kK; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(chunk_addr(ks, row, 2 * j + (i >> 1), p.region_stride), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          mma_16816<kBF16>(s[nt], a0, a1, a2, a3, qf[nt][j][0], qf[nt][j][1]);
      }
    }

    // ---- online softmax over the tile's 16 tokens (rows g, g+8), heads 2*t4 + {0,1}
    const bool ok_lo = kFull || ((valid >> g) & 1u), ok_hi = kFull || ((valid >> (g + 8)) & 1u);
    uint32_t pb[kNT][2][kSplitP ? 2 : 1];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      float pr[4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float a = ok_lo ? s[nt][hh] * score_scale : -INFINITY;
        const float b = ok_hi ? s[nt][2 + hh] * score_scale : -INFINITY;
        float mx = fmaxf(a, b);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m[nt][hh], mx);
        const float ref = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m[nt][hh] - ref);
        m[nt][hh] = mnew;
        pr[hh] = ex2(a - ref);
        pr[2 + hh] = ex2(b - ref);
        l[nt][hh] = l[nt][hh] * alpha + pr[hh] + pr[2 + hh];
#pragma unroll
        for (int j = 0; j < kK; ++j) {
          o[nt][j][hh] *= alpha;
          o[nt][j][2 + hh] *= alpha;
        }
      }
      // P^T as the B operand: rows (tokens g | g+8) x cols (heads 2t4, 2t4+1) -> transpose
      if constexpr (kSplitP) {
        const uint32_t h0 = pack2<kBF16>(pr[0], pr[1]);
        const uint32_t h1 = pack2<kBF16>(pr[2], pr[3]);
        const float2 r0f = unpack2<kBF16>(h0), r1f = unpack2<kBF16>(h1);
        const uint32_t lo0 = pack2<kBF16>(pr[0] - r0f.x, pr[1] - r0f.y);
        const uint32_t lo1 = pack2<kBF16>(pr[2] - r1f.x, pr[3] - r1f.y);
        pb[nt][0][0] = movmatrix_t(h0);
        pb[nt][1][0] = movmatrix_t(h1);
        pb[nt][0][1] = movmatrix_t(lo0);
        pb[nt][1][1] = movmatrix_t(lo1);
      } else {
        pb[nt][0][0] = movmatrix_t(pack2<false>(pr[0], pr[1]));
        pb[nt][1][0] = movmatrix_t(pack2<false>(pr[2], pr[3]));
      }
    }

    // masks of the value rows this lane feeds: tokens (2t4, 2t4+1) and (2t4+8, 2t4+9)
    uint32_t mask01 = 0xffffffffu, mask23 = 0xffffffffu;
    if (!kFull && valid != 0xffffu) {
      mask01 = (((valid >> (2 * t4)) & 1u) ? 0x0000ffffu : 0u) |
               (((valid >> (2 * t4 + 1)) & 1u) ? 0xffff0000u : 0u);
      mask23 = (((valid >> (2 * t4 + 8)) & 1u) ? 0x0000ffffu : 0u) |
               (((valid >> (2 * t4 + 9)) & 1u) ? 0xffff0000u : 0u);
    }

    // ---- O^T += V^T P^T
    if constexpr (kFp8) {
      // lane reads 16-byte chunk g of token rows 2t4, 2t4+1, 2t4+8, 2t4+9 and interleaves the
      // token pairs: m-tile j row g <-> d = 16g + 2j, row g+8 <-> d = 16g + 2j + 1
      uint32_t va[2][16];
#pragma unroll
      for (int pair = 0; pair < 2; ++pair) {
        const StageRow ra = stage_row(r0 + 2 * t4 + 8 * pair, p.log2_srows, Gm::kRegions, p.region_stride);
        const StageRow rb = stage_row(r0 + 2 * t4 + 8 * pair + 1, p.log2_srows, Gm::kRegions, p.region_stride);
        const uint4 x = lds128(chunk_addr(vs, ra, g, p.region_stride));
        const uint4 y = lds128(chunk_addr(vs, rb, g, p.region_stride));
        const uint32_t xa[4] = {x.x, x.y, x.z, x.w};
        const uint32_t ya[4] = {y.x, y.y, y.z, y.w};
        const uint32_t msk = pair ? mask23 : mask01;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t lo = prmt(xa[w], ya[w], 0x5140u);
          const uint32_t hi = prmt(xa[w], ya[w], 0x7362u);
          va[pair][4 * w + 0] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo & 0xffffu));
          va[pair][4 * w + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo >> 16));
          va[pair][4 * w + 2] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi & 0xffffu));
          va[pair][4 * w + 3] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi >> 16));
          if constexpr (!kFull) {
#pragma unroll
            for (int e = 0; e < 4; ++e) va[pair][4 * w + e] &= msk;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kK; ++j) {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          mma_16816<false>(o[nt][j], va[0][2 * j], va[0][2 * j + 1], va[1][2 * j],
                           va[1][2 * j + 1], pb[nt][0][0], pb[nt][1][0]);
      }
    } else {
      const int i = lane >> 3;
      const StageRow row =
          stage_row(r0 + (lane & 7) + 8 * (i >> 1), p.log2_srows, Gm::kRegions, p.region_stride);
#pragma unroll
      for (int j = 0; j < kK; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(chunk_addr(vs, row, 2 * j + (i & 1), p.region_stride), a0, a1, a2, a3);
        if constexpr (!kFull) {
          a0 &= mask01;
          a1 &= mask01;
          a2 &= mask23;
          a3 &= mask23;
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          mma_16816<kBF16>(o[nt][j], a0, a1, a2, a3, pb[nt][0][0], pb[nt][1][0]);
          mma_16816<kBF16>(o[nt][j], a0, a1, a2, a3, pb[nt][0][1], pb[nt][1][1]);
        }
      }
    }
  }

  __device__ void publish(float* mrg_o, float2* mrg_ml, int cw, int lane) {
    (void)lane;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float lsum = l[nt][hh];
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
        const int n = nt * 8 + 2 * t4 + hh;
        if (n < G) {
          float* dst = mrg_o + (cw * G + n) * D;
#pragma unroll
          for (int j = 0; j < kK; ++j) {
            if constexpr (kFp8) {
              dst[16 * g + 2 * j] = o[nt][j][hh];
              dst[16 * g + 2 * j + 1] = o[nt][j][2 + hh];
            } else {
              dst[16 * j + g] = o[nt][j][hh];
              dst[16 * j + g + 8] = o[nt][j][2 + hh];
            }
          }
          if (g == 0) mrg_ml[cw * G + n] = make_float2(m[nt][hh], lsum);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void store_out(void* out, size_t idx, float v, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// Combine the ns split partials of one (sequence, query head) with one warp: lane i holds the
// (max, sum) pair of split i of each pass of 32, the weights w_i = 2^(m_i - m*) / sum_j
// 2^(m_j - m*) l_j are formed with shuffles, then out = sum_i w_i * acc_i with float4 loads
// (lane c owns columns 4c..4c+3). Used for more than 32 splits.
template <int D>
__device__ void combine_head_long(const DecodeParams& p, int ns, size_t head, int lane, bool out_bf16) {
  constexpr int kVec = D / 4;
  const size_t slot0 = head * p.max_splits;
  float m_own = -INFINITY, l_own = 0.f;  // split `lane` (first pass of 32)
  if (lane < ns) {
    const float2 ml = __ldcg(&p.part_ml[slot0 + lane]);
    m_own = ml.x;
    l_own = ml.y;
  }
  float mstar = m_own;
  for (int i = lane + 32; i < ns; i += 32) mstar = fmaxf(mstar, __ldcg(&p.part_ml[slot0 + i].x));
  for (int off = 16; off; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  const float4* src = reinterpret_cast<const float4*>(p.part_o + slot0 * D);
  for (int i0 = 0; i0 < ns; i0 += 32) {
    const int cnt = min(32, ns - i0);
    float e = 0.f;
    if (lane < cnt && mstar != -INFINITY) {
      float m = m_own, l = l_own;
      if (i0 > 0) {
        const float2 ml = __ldcg(&p.part_ml[slot0 + i0 + lane]);
        m = ml.x;
        l = ml.y;
      }
      e = ex2(m - mstar);
      den = fmaf(e, l, den);
    }
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float ej = __shfl_sync(0xffffffffu, e, j);
      if (lane < kVec) {
        const float4 v = __ldcg(src + static_cast<size_t>(i0 + j) * kVec + lane);
        acc.x = fmaf(ej, v.x, acc.x);
        acc.y = fmaf(ej, v.y, acc.y);
        acc.z = fmaf(ej, v.z, acc.z);
        acc.w = fmaf(ej, v.w, acc.w);
      }
    }
  }
  for (int off = 16; off; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  if (lane < kVec) {
    const size_t o = head * D + 4 * lane;
    store_out(p.out, o, acc.x * inv, out_bf16);
    store_out(p.out, o + 1, acc.y * inv, out_bf16);
    store_out(p.out, o + 2, acc.z * inv, out_bf16);
    store_out(p.out, o + 3, acc.w * inv, out_bf16);
  }
}

// Combine of up to 32 split partials for kH consecutive query heads of one kv group (they share
// the split count), by one warp: out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i with
// M = max_i m_i. The (max, sum) pairs and the first kB * (32 / (D / 4)) partial rows of every
// head are loaded at once, so a warp's heads cost about one L2 round trip. Split i's pair sits
// in lane i; lane c covers float4 column c % (D / 4) of splits c / (D / 4), c / (D / 4) +
// 32 / (D / 4), ...
template <int D, int kH>
__device__ void combine_heads(const DecodeParams& p, int ns, size_t head0, int lane, bool out_bf16) {
  constexpr int kVec = D / 4;
  constexpr int kRows = 32 / kVec;
  constexpr int kB = 8;
  const int col = lane % kVec, row = lane / kVec;
  float2 ml[kH];
  float4 v[kH][kB], acc[kH];
  float M[kH], w[kH], den[kH];
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    const size_t slot0 = (head0 + h) * p.max_splits;
    ml[h] = lane < ns ? __ldcg(&p.part_ml[slot0 + lane]) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int j = k * kRows + row;
      v[h][k] = j < ns ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (slot0 + j) * D) + col)
                       : zero;
    }
    acc[h] = zero;
  }
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    M[h] = ml[h].x;
    for (int off = 16; off; off >>= 1) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], off));
    w[h] = (lane < ns && M[h] != -INFINITY) ? ex2(ml[h].x - M[h]) : 0.f;
    den[h] = w[h] * ml[h].y;
    for (int off = 16; off; off >>= 1) den[h] += __shfl_xor_sync(0xffffffffu, den[h], off);
  }
  for (int j0 = 0; j0 < ns; j0 += kB * kRows) {
    if (j0 > 0) {
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        const size_t slot0 = (head0 + h) * p.max_splits;
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          const int j = j0 + k * kRows + row;
          v[h][k] = j < ns ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (slot0 + j) * D) + col)
                           : zero;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kH; ++h) {
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        const int j = j0 + k * kRows + row;
        const float wj = __shfl_sync(0xffffffffu, w[h], j & 31);
        if (j < ns) {
          acc[h].x = fmaf(wj, v[h][k].x, acc[h].x);
          acc[h].y = fmaf(wj, v[h][k].y, acc[h].y);
          acc[h].z = fmaf(wj, v[h][k].z, acc[h].z);
          acc[h].w = fmaf(wj, v[h][k].w, acc[h].w);
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    if (kRows == 2) {
      acc[h].x += __shfl_xor_sync(0xffffffffu, acc[h].x, 16);
      acc[h].y += __shfl_xor_sync(0xffffffffu, acc[h].y, 16);
      acc[h].z += __shfl_xor_sync(0xffffffffu, acc[h].z, 16);
      acc[h].w += __shfl_xor_sync(0xffffffffu, acc[h].w, 16);
    }
    const float inv = den[h] > 0.f ? 1.f / den[h] : 0.f;
    if (lane < kVec) {
      const size_t o = (head0 + h) * D + 4 * col;
      store_out(p.out, o, acc[h].x * inv, out_bf16);
      store_out(p.out, o + 1, acc[h].y * inv, out_bf16);
      store_out(p.out, o + 2, acc[h].z * inv, out_bf16);
      store_out(p.out, o + 3, acc[h].w * inv, out_bf16);
    }
  }
}

__device__ __forceinline__ int row_of(const int (&rows)[4], int b) {
  return b == 0 ? rows[0] : b == 1 ? rows[1] : b == 2 ? rows[2] : rows[3];
}

template <int KV, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    pa_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeParams p) {
  using Gm = Geom<KV, D>;
  constexpr bool kMma = G >= 4;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  constexpr int kFirstConsumer = 1 + kProducerWarps;  // warp index of consumer 0
  const bool qbf = p.q_bf16 != 0;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // ring of stages starts here
  uint8_t* bp = smem_raw + (base - raw);
  float* mrg_o = reinterpret_cast<float*>(bp + p.off_merge);
  float2* mrg_ml = reinterpret_cast<float2*>(bp + p.off_merge + kConsumerWarps * G * D * 4);
  uint16_t* qbuf = reinterpret_cast<uint16_t*>(bp + p.off_q);  // [kItemSlots][G * D]
  uint64_t* bar = reinterpret_cast<uint64_t*>(bp + p.off_bar);
  uint64_t* full = bar;                       // [kMaxStages] stage landed
  uint64_t* empty = bar + kMaxStages;         // [kMaxStages] stage consumed
  uint64_t* qfull = bar + 2 * kMaxStages;     // [kItemSlots] item descriptor and table written
  uint64_t* qempty = qfull + kItemSlots;      // [kItemSlots] slot released by producers + consumers
  uint64_t* qland = qempty + kItemSlots;      // [kItemSlots] item queries landed (bulk copy)
  uint64_t* sorted = qland + kItemSlots;      // [1] part-2 order written by the consumer warps
  uint32_t* meta = reinterpret_cast<uint32_t*>(bp + p.off_meta);     // [kMaxStages] valid tokens
  ItemDesc* items = reinterpret_cast<ItemDesc*>(bp + p.off_items);  // [kItemSlots]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(items + kItemSlots);
  int* tbl = reinterpret_cast<int*>(bp + p.off_tbl);      // [kItemSlots][tbl_stride]
  int* pf1 = reinterpret_cast<int*>(bp + p.off_scan);  // [num_seqs + 1] full-split items
  int* pf2 = pf1 + p.num_seqs + 1;                       // [num_seqs + 1] last-split items
  int* order2 = pf2 + p.num_seqs + 1;                    // [num_seqs] part-2 sequence order
  int* wsum = order2 + p.num_seqs;                       // [2 * kScanWarps] warp totals
  int* wcnt = wsum + 2 * kScanWarps;                     // [kScanWarps][kRemBuckets]
  int* bstart = wcnt + kScanWarps * kRemBuckets;         // [kRemBuckets] next free position
  int* bcnt = bstart + kRemBuckets;                      // [kRemBuckets] sequences per bucket

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.num_seqs, Hkv = p.num_kv_heads, B = p.block_size, S = p.split_tokens;
  const int st_tokens = p.stage_tokens;

  // ---- prologue: the work list. Part 1 holds every full-length split of every sequence
  // (sequence order, then kv head, then split); part 2 the shorter last split of each sequence
  // whose context is not a multiple of split_tokens, longest first (a stable counting sort
  // over kRemBuckets size classes), so the list ends with the smallest items and the CTAs run
  // out of work at nearly the same time. pf1/pf2 are per-sequence prefix sums of item counts.
  // Every CTA builds the same list.
  auto rem_bucket = [&](int L) -> int {  // size class of the last split, -1 if it is full/empty
    const bool bad = L < 0 || L > p.max_ctx || L > p.max_blocks * B;
    const int r = (bad || L == 0) ? 0 : L % S;
    return r == 0 ? -1 : kRemBuckets - 1 - static_cast<int>((static_cast<int64_t>(r - 1) * kRemBuckets) / S);
  };
  if (tid < kScanWarps * kRemBuckets) wcnt[tid] = 0;
  if (tid < kRemBuckets) bcnt[tid] = 0;
  __syncthreads();
  {
    const int per = (N + kDecodeThreads - 1) / kDecodeThreads;
    const int s0 = min(N, tid * per), s1 = min(N, s0 + per);
    int c1 = 0, c2 = 0;
    for (int s = s0; s < s1; ++s) {
      const int L = __ldg(p.ctx_lens + s);
      const bool bad = L < 0 || L > p.max_ctx || L > p.max_blocks * B;
      const int nfull = (bad || L == 0) ? 0 : L / S;
      const int rem = (bad || L == 0) ? 0 : (L % S != 0);
      pf1[s] = nfull * Hkv;
      pf2[s] = rem * Hkv;
      if (rem) atomicAdd(&bcnt[rem_bucket(L)], 1);
      c1 += nfull * Hkv;
      c2 += rem * Hkv;
      if ((bad || L == 0) && (s % gridDim.x) == blockIdx.x) {
        if (bad) flag_error(p.err, kErrCtxLen);
        const size_t row0 = static_cast<size_t>(s) * p.num_q_heads * D;
        for (int i = 0; i < p.num_q_heads * D; ++i) store_out(p.out, row0 + i, 0.f, qbf);
      }
    }
    if (tid == 0) {
      *abort_flag = 0;
      for (int s = 0; s < p.stages; ++s) {
        mbar_init(smem_addr(full + s), 1);
        mbar_init(smem_addr(empty + s), 1);
      }
      for (int b = 0; b < kItemSlots; ++b) {
        mbar_init(smem_addr(qfull + b), 1);
        mbar_init(smem_addr(qempty + b), kProducerWarps + kConsumerWarps);
        mbar_init(smem_addr(qland + b), 1);
      }
      mbar_init(smem_addr(sorted), 1);
      fence_barrier_init();
    }
    // block-wide exclusive scan of (c1, c2): warp scans, then a scan of the warp totals
    constexpr int kWarps = kDecodeThreads / 32;
    int i1 = c1, i2 = c2;
    for (int off = 1; off < 32; off <<= 1) {
      const int t1 = __shfl_up_sync(0xffffffffu, i1, off);
      const int t2 = __shfl_up_sync(0xffffffffu, i2, off);
      if (lane >= off) {
        i1 += t1;
        i2 += t2;
      }
    }
    if (lane == 31) {
      wsum[2 * warp] = i1;
      wsum[2 * warp + 1] = i2;
    }
    __syncthreads();
    if (warp == 0) {
      const int v1 = lane < kWarps ? wsum[2 * lane] : 0;
      const int v2 = lane < kWarps ? wsum[2 * lane + 1] : 0;
      int u1 = v1, u2 = v2;
      for (int off = 1; off < 32; off <<= 1) {
        const int t1 = __shfl_up_sync(0xffffffffu, u1, off);
        const int t2 = __shfl_up_sync(0xffffffffu, u2, off);
        if (lane >= off) {
          u1 += t1;
          u2 += t2;
        }
      }
      if (lane < kWarps) {
        wsum[2 * lane] = u1 - v1;
        wsum[2 * lane + 1] = u2 - v2;
      }
      if (lane == kWarps - 1) {
        pf1[N] = u1;
        pf2[N] = u2;
      }
    } else if (warp == 1) {  // bucket b (0 = longest) starts after the sequences of buckets < b
      const int v = bcnt[lane];
      int u = v;
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, u, off);
        if (lane >= off) u += t;
      }
      bstart[lane] = u - v;
    }
    __syncthreads();
    int run1 = wsum[2 * warp] + i1 - c1, run2 = wsum[2 * warp + 1] + i2 - c2;
    for (int s = s0; s < s1; ++s) {
      const int a1 = pf1[s], a2 = pf2[s];
      pf1[s] = run1;
      pf2[s] = run2;
      run1 += a1;
      run2 += a2;
    }
    __syncthreads();
  }
  const int items1 = pf1[N];
  const int total_items = items1 + pf2[N];

  if (warp == 0) {
    // ------------------------------------------------------------------ scheduler warp
    // Takes items from the global counter and fills the item slots: descriptor, the item's
    // block-table slice (validated) and, by bulk copy, its queries.
    const uint32_t qbytes = static_cast<uint32_t>(G * D * 2);
    bool have_order = false;  // lane 0: the consumers' part-2 order is complete
    int last_q[kItemSlots];   // lane 0: item number of the last query copy into each slot
    for (int b = 0; b < kItemSlots; ++b) last_q[b] = -1;
    for (uint32_t it = 0;; ++it) {
      const int slot = it % kItemSlots;
      if (it >= kItemSlots &&
          !mbar_wait_bounded(smem_addr(qempty + slot), ((it / kItemSlots) - 1) & 1, p.wait_ns)) {
        if (lane == 0) {
          flag_error(p.err, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      int item = 0, seq = 0;
      if (lane == 0) {
        // the first item of CTA b is item b; the counter hands out the rest
        item = it == 0 ? static_cast<int>(blockIdx.x)
                       : static_cast<int>(gridDim.x + fetch_ticket(p.counters, p.launch_id));
        if (item >= items1 && item < total_items && !have_order) {
          have_order = mbar_wait_bounded(smem_addr(sorted), 0, p.wait_ns);
          if (!have_order) {
            flag_error(p.err, kErrTimeout);
            *abort_flag = 1;
          }
        }
        if (item < items1) {
          int lo = 0, hi = N - 1;  // largest s with pf1[s] <= item
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pf1[mid] <= item) lo = mid; else hi = mid - 1;
          }
          seq = lo;
        } else if (item < total_items) {
          seq = order2[(item - items1) / Hkv];
        }
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      seq = __shfl_sync(0xffffffffu, seq, 0);
      ItemDesc& d = items[slot];
      if (item >= total_items || *abort_flag) {
        if (lane == 0) {
          d.seq = -1;
          mbar_arrive(smem_addr(qfull + slot));
        }
        break;
      }
      const int L = __ldg(p.ctx_lens + seq);
      const int nfull = (pf1[seq + 1] - pf1[seq]) / Hkv;
      const int nsplit = nfull + (pf2[seq + 1] - pf2[seq]) / Hkv;
      int kvh, split;
      if (item < items1) {
        const int li = item - pf1[seq];
        kvh = li / nfull;
        split = li % nfull;
      } else {
        kvh = (item - items1) % Hkv;
        split = nfull;
      }
      const int tok0 = split * S, tok_end = min(L, tok0 + S);
      // the row of every copy unit (srows rows of one block's tile for kv head kvh), so the
      // producers only look it up: unit u starts at token tok0 + u * srows
      const int blk0 = tok0 >> p.log2_block;
      const int nunits = (tok_end - tok0 + (1 << p.log2_srows) - 1) >> p.log2_srows;
      const int32_t* trow = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + blk0;
      int* slot_tbl = tbl + slot * p.tbl_stride;
      for (int u = lane; u < nunits; u += 32) {
        const int rel = u << p.log2_srows;
        int ph = __ldg(trow + (rel >> p.log2_block));
        if (ph < 0 || ph >= p.num_blocks) {
          flag_error(p.err, kErrBlockId);
          slot_tbl[u] = -1;
        } else {
          slot_tbl[u] = (ph * Hkv + kvh) * B + (rel & (B - 1));
        }
      }
      __syncwarp();
      if (lane == 0) {
        d.seq = seq;
        d.kvh = kvh;
        d.split = split;
        d.nsplit = nsplit;
        d.ntiles = (tok_end - tok0 + st_tokens - 1) / st_tokens;
        d.tok0 = tok0;
        d.tok_end = tok_end;
        d.nunits = nunits;
        // descriptor and table for the producers now, the queries for the consumers on landing
        mbar_arrive(smem_addr(qfull + slot));
        const uint32_t ql = smem_addr(qland + slot);
        mbar_arrive_expect_tx(ql, qbytes);
        bulk_copy_g2s(smem_addr(qbuf + slot * G * D),
                      static_cast<const uint16_t*>(p.q) +
                          (static_cast<size_t>(seq) * p.num_q_heads + kvh * G) * D,
                      qbytes, ql);
        last_q[slot] = static_cast<int>(it);
      }
    }
    // No query copy may still be landing when the CTA exits. Normally the consumers have waited
    // for every one; after an abort they may not have. The last copy into a slot completes the
    // slot's barrier phase of that item, and no later phase was started.
    if (lane == 0) {
      for (int b = 0; b < kItemSlots; ++b)
        if (last_q[b] >= 0)
          mbar_wait_bounded(smem_addr(qland + b), (static_cast<uint32_t>(last_q[b]) / kItemSlots) & 1,
                            kDrainLimitNs);
    }
  } else if (warp <= kProducerWarps) {
    // ------------------------------------------------------------------ producer warps
    // Producer pw issues the tiles g = pw (mod kProducerWarps) of the CTA's tile sequence.
    // Several issuing warps keep enough copies in flight: one warp alone streams far below
    // the per-SM share of HBM bandwidth.
    const int pw = warp - 1;
    // K/V tiles are streamed once (shared-prompt blocks are re-read within microseconds by the
    // neighbouring items of the other group members), so they are marked evict-first in L2.
    const uint64_t pol = policy_evict_first();
    if (lane == 0 && pw == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    // A stage holds bps copies of srows rows each: whole blocks when blocks are at most a stage
    // (bps = 1, 2 or 4), else one part of one block (bps = 1, srows = stage tokens).
    const int srows = 1 << p.log2_srows;
    const uint32_t tile_bytes = static_cast<uint32_t>(2 * Gm::kRegions * srows * 128);
    const int bps = st_tokens >> p.log2_srows;
    uint32_t g0 = 0;                            // CTA tile index of the item's first tile
    bool ok = true;
    uint32_t issued_last = 0, any = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = it % kItemSlots;
      if (!mbar_wait_bounded(smem_addr(qfull + slot), (it / kItemSlots) & 1, p.wait_ns)) {
        ok = false;
        break;
      }
      const ItemDesc d = items[slot];
      if (d.seq < 0) break;
      const int* slot_tbl = tbl + slot * p.tbl_stride;
      int t = (pw - static_cast<int>(g0 % kProducerWarps) + kProducerWarps) % kProducerWarps;
      for (; t < d.ntiles; t += kProducerWarps) {
        const uint32_t g = g0 + t;
        const int s = static_cast<int>(g % p.stages);
        if (g >= static_cast<uint32_t>(p.stages) &&
            !mbar_wait_bounded(smem_addr(empty + s), ((g / p.stages) - 1) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        uint32_t valid = 0, bytes = 0;
        int rows[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          rows[b] = -1;
          const int u = t * bps + b;  // copy unit b of stage t
          if (b < bps && u < d.nunits) {
            const int row = slot_tbl[u];
            if (row >= 0) {
              rows[b] = row;
              bytes += tile_bytes;
              const int r0 = b * srows;
              const int n = min(srows, d.tok_end - (d.tok0 + t * st_tokens + r0));
              valid |= (n >= 32 ? 0xffffffffu : ((1u << n) - 1u)) << r0;
            }
          }
        }
        const uint32_t fb = smem_addr(full + s);
        if (lane == 0) {
          meta[s] = valid;
          mbar_arrive_expect_tx(fb, bytes);
        }
        __syncwarp();
        {  // one lane per copy: (block b, K|V, column region c)
          constexpr int kOps = 2 * Gm::kRegions;
          const int b = lane / kOps, kv = (lane / Gm::kRegions) & 1, c = lane % Gm::kRegions;
          if (b < bps && row_of(rows, b) >= 0) {
            const uint32_t off = static_cast<uint32_t>(2 * s * p.stage_bytes + kv * p.stage_bytes +
                                                       (b * Gm::kRegions + c) * p.region_stride);
            tma_load_2d(base + off, kv ? &vmap : &kmap, c * Gm::kColsPerRegion, row_of(rows, b),
                        fb, pol);
          }
        }
        issued_last = g;
        any = 1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(qempty + slot));
      if (!ok) break;
      g0 += d.ntiles;
    }
    if (!ok) {
      if (lane == 0) {
        flag_error(p.err, kErrTimeout);
        *abort_flag = 1;
      }
      // nothing this warp issued may still be landing in shared memory when the CTA exits
      if (any) {
        const uint32_t span = static_cast<uint32_t>(p.stages);
        const uint32_t from = issued_last >= span ? issued_last - span + 1 : 0u;
        for (uint32_t g = from; g <= issued_last; ++g)
          if (g % kProducerWarps == static_cast<uint32_t>(pw))
            mbar_wait_bounded(smem_addr(full + (g % p.stages)), (g / p.stages) & 1, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------------ consumer warps
    const int cw = warp - kFirstConsumer;
    const int ctid = tid - kFirstConsumer * 32;
    Consumer<KV, D, G, kMma> c;
    // Part-2 order (the scheduler needs it only once part 1 is handed out): chunks of
    // kConsumerThreads sequences; a sequence's position is its bucket's start, plus the
    // bucket's sequences in earlier consumer warps of the chunk, plus those in earlier lanes.
    for (int c0 = 0; c0 < N; c0 += kConsumerThreads) {
      const int s = c0 + ctid;
      const int b = s < N ? rem_bucket(__ldg(p.ctx_lens + s)) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, b);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (b >= 0 && rank == 0) wcnt[cw * kRemBuckets + b] = __popc(peers);
      bar_sync(1, kConsumerThreads);
      if (b >= 0) {
        int pos = bstart[b] + rank;
        for (int w = 0; w < cw; ++w) pos += wcnt[w * kRemBuckets + b];
        order2[pos] = s;
      }
      bar_sync(1, kConsumerThreads);
      if (ctid < kRemBuckets) {
        int add = 0;
        for (int w = 0; w < kConsumerWarps; ++w) {
          add += wcnt[w * kRemBuckets + ctid];
          wcnt[w * kRemBuckets + ctid] = 0;
        }
        bstart[ctid] += add;
      }
      bar_sync(1, kConsumerThreads);
    }
    if (ctid == 0) mbar_arrive(smem_addr(sorted));
    uint32_t g0 = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = it % kItemSlots;
      bool got = mbar_wait_bounded(smem_addr(qfull + slot), (it / kItemSlots) & 1, p.wait_ns);
      const ItemDesc d = items[slot];
      if (got && d.seq >= 0)
        got = mbar_wait_bounded(smem_addr(qland + slot), (it / kItemSlots) & 1, p.wait_ns);
      if (bar_or(kConsumerThreads, !got)) {  // every consumer warp leaves together
        if (ctid == 0) {
          flag_error(p.err, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      if (d.seq < 0) break;
      c.init(qbuf + slot * G * D, qbf, lane);
      float score_scale = p.score_scale;
      if constexpr (kMma && KV == kKvE4M3) score_scale *= c.qexp;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(qempty + slot));

      bool ok = true;
      for (int t = cw; t < d.ntiles; t += kConsumerWarps) {
        const uint32_t g = g0 + t;
        const int s = static_cast<int>(g % p.stages);
        if (!mbar_wait_bounded(smem_addr(full + s), (g / p.stages) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t valid = meta[s];
        const uint32_t ks = base + static_cast<uint32_t>(2 * s * p.stage_bytes);
        const uint32_t vs = ks + static_cast<uint32_t>(p.stage_bytes);
        for (int sub = 0; sub < st_tokens; sub += 16) {
          const uint32_t v16 = (valid >> sub) & 0xffffu;
          if (v16) c.tile(p, ks, vs, sub, v16, score_scale);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(empty + s));
      }

      // merge the consumer warps' states for this item and write it out
      c.publish(mrg_o, mrg_ml, cw, lane);
      bar_sync(1, kConsumerThreads);
      const size_t head0 = static_cast<size_t>(d.seq) * p.num_q_heads + d.kvh * G;
      for (int idx = ctid; idx < G * D; idx += kConsumerThreads) {
        const int n = idx / D, dd = idx % D;
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mstar = fmaxf(mstar, mrg_ml[w * G + n].x);
        float num = 0.f, den = 0.f;
        if (mstar != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float2 ml = mrg_ml[w * G + n];
            const float wgt = ex2(ml.x - mstar);
            num = fmaf(wgt, mrg_o[(w * G + n) * D + dd], num);
            den = fmaf(wgt, ml.y, den);
          }
        }
        if (d.nsplit == 1) {
          store_out(p.out, (head0 + n) * D + dd, den > 0.f ? num / den * p.v_scale : 0.f, qbf);
        } else {
          const size_t slot_i = (head0 + n) * p.max_splits + d.split;
          p.part_o[slot_i * D + dd] = num * p.v_scale;
          if (dd == 0) p.part_ml[slot_i] = make_float2(mstar, den);
        }
      }
      if (bar_or(kConsumerThreads, !ok || *abort_flag)) {
        if (ctid == 0) {
          flag_error(p.err, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      g0 += d.ntiles;
    }
  }

  // ---- split-K combine. The kernel is a cooperative launch (every CTA resident), so after one
  // grid-wide barrier all partials are in memory and the CTAs combine them: one warp per
  // (sequence, query head) with more than one split. One fence per CTA instead of one per item.
  __syncthreads();
  if (p.max_splits > 1) {
    if (tid == 0) {
      __threadfence();  // this CTA's partials are visible to the whole GPU before it arrives
      if (static_cast<int>(blockIdx.x) != p.stall_cta) fetch_ticket(p.counters + 2, p.launch_id);
      const unsigned long long* ctr = p.counters + 2;
      const unsigned long long start = global_ns();
      bool ok = true;
      for (uint32_t i = 0;; ++i) {
        const unsigned long long v = *reinterpret_cast<const volatile unsigned long long*>(ctr);
        if ((v >> 32) == p.launch_id && static_cast<uint32_t>(v) >= gridDim.x) break;
        if ((i & 63u) == 63u && global_ns() - start > p.wait_ns) {
          ok = false;
          break;
        }
      }
      __threadfence();
      if (!ok) {
        flag_error(p.err, kErrTimeout);
        *abort_flag = 1;
      }
    }
    __syncthreads();
    if (!*abort_flag) {
      // one warp per kH query heads of a kv group (they share the sequence's split count);
      // consecutive units go to different CTAs
      constexpr int kH = G < 2 ? G : 2;
      const int nwarps = kDecodeThreads / 32;
      const int units = N * (p.num_q_heads / kH);
      for (int u = warp * gridDim.x + blockIdx.x; u < units; u += gridDim.x * nwarps) {
        const size_t head0 = static_cast<size_t>(u) * kH;
        const int seq = static_cast<int>(head0 / p.num_q_heads);
        const int ns = (pf1[seq + 1] - pf1[seq] + pf2[seq + 1] - pf2[seq]) / Hkv;  // 0: none
        if (ns > 32) {
          for (int h = 0; h < kH; ++h) combine_head_long<D>(p, ns, head0 + h, lane, qbf);
        } else if (ns > 1) {
          combine_heads<D, kH>(p, ns, head0, lane, qbf);
        }
      }
    }
  }

  // ---- the last CTA to finish clears the work counters for the next launch
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t done = fetch_ticket(p.counters + 1, p.launch_id);
    if (done == gridDim.x - 1) {
      atomicExch(p.counters, 0ull);
      atomicExch(p.counters + 1, 0ull);
      atomicExch(p.counters + 2, 0ull);
    }
  }
}

}  // namespace pa

namespace pa {

// Host: record of (kernel, device) pairs already opted in to the full shared memory.
inline std::mutex& opt_in_mutex() {
  static std::mutex m;
  return m;
}
inline std::set<std::pair<const void*, int>>& opt_in_set() {
  static std::set<std::pair<const void*, int>> s;
  return s;
}
inline bool smem_opted_in(const void* fn, int dev) {
  std::lock_guard<std::mutex> g(opt_in_mutex());
  return opt_in_set().count({fn, dev}) != 0;
}
inline void mark_smem_opted_in(const void* fn, int dev) {
  std::lock_guard<std::mutex> g(opt_in_mutex());
  opt_in_set().insert({fn, dev});
}

// Host: launch the decode kernel instantiation for (KV, head_dim, group).
template <int KV>
cudaError_t launch_decode_kv(int head_dim, int group, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, const DecodeParams& p, dim3 grid,
                             size_t smem, cudaStream_t stream) {
  decltype(&pa_decode_kernel<KV, 128, 1>) fn = nullptr;
#define PA_DECODE_CASE(D_, G_) \
  if (head_dim == D_ && group == G_) fn = &pa_decode_kernel<KV, D_, G_>;
  PA_DECODE_CASE(128, 1)
  PA_DECODE_CASE(128, 2)
  PA_DECODE_CASE(128, 4)
  PA_DECODE_CASE(128, 8)
  PA_DECODE_CASE(128, 16)
  if constexpr (KV != kKvE4M3) {
    PA_DECODE_CASE(64, 1)
    PA_DECODE_CASE(64, 2)
    PA_DECODE_CASE(64, 4)
    PA_DECODE_CASE(64, 8)
    PA_DECODE_CASE(64, 16)
  }
#undef PA_DECODE_CASE
  if (fn == nullptr) return cudaErrorInvalidValue;
  // Opt in to the full shared memory once per device (not per call, so that launches can be
  // captured into CUDA graphs without extra API calls).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!smem_opted_in(reinterpret_cast<const void*>(fn), dev)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    mark_smem_opted_in(reinterpret_cast<const void*>(fn), dev);
  }
  // Cooperative launch: the combine phase waits on every CTA, so all must be resident at once.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, kmap, vmap, p);
}

}  // namespace pa
