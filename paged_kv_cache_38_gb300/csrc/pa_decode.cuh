// pa_decode.cuh - paged decode attention kernels for sm_103a (templates; instantiated per KV dtype).
//
// Method: "Efficient Memory Management for Large Language Model Serving with PagedAttention"
// (paper summary page), paragraph on the PagedAttention kernel: the keys of logical block j sit
// in a physical block found through the sequence's block table; the kernel fetches every block
// wherever it is stored, scores the query against it and combines the values, and the result
// equals ordinary attention. "Continuous Batching and PagedAttention", section "The block table
// is a page table": the kernel gathers through the table instead of striding.
//
// GB300 design (one CTA per (context split, kv head, sequence)):
//   * warp 0 is the producer: one lane walks the split's block-table slice (read once into shared
//     memory, out-of-pool ids masked and flagged) and issues 2-D TMA tensor copies of each
//     (block, kv head) tile of K and V into a ring of shared-memory stages, 128-byte swizzled,
//     completing on per-stage mbarriers;
//   * warps 1..4 are consumers: stage t is consumed by warp t % 4, each with its own online
//     softmax state (running max in log2 units, running sum, fp32 accumulator);
//   * group size G <= 2: warp-shuffle dot products (CUDA cores), one token row per lane group;
//     G >= 4: the GQA group makes each 16-token tile a small dense contraction, done with
//     mma.sync m16n8k16 (S^T = K Q^T with the G query heads as the N dimension, then
//     O^T += V^T P^T), fp32 accumulation;
//   * the four consumer states are merged in shared memory; one split writes the output
//     directly, several splits write fp32 partials that pa_reduce_kernel combines.
#pragma once

#include "pa_device.cuh"

namespace pa {

enum KvKind { kKvF16 = 0, kKvBF16 = 1, kKvE4M3 = 2 };

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (1 + kConsumerWarps);
constexpr int kMaxStages = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  float* part_o;    // [num_seqs][num_q_heads][max_splits][D] unnormalised, v_scale applied
  float2* part_ml;  // [num_seqs][num_q_heads][max_splits] (max score in log2 units, weight sum)
  int32_t* err;
  int num_seqs, num_q_heads, num_kv_heads;
  int block_size, log2_block, num_blocks, max_blocks, max_ctx;
  int split_tokens;   // tokens per split, a multiple of max(16, block_size)
  int max_splits;     // ceil(max_ctx / split_tokens)
  int stages;         // shared-memory ring depth, a multiple of kConsumerWarps
  int region_stride;  // bytes of one 128-byte-wide column region of one block in a stage
  int stage_bytes;    // bytes of K (or V) in one stage
  int ctl_offset;     // offset of the barriers / table area from the aligned smem base
  float score_scale;  // scale * k_scale * log2(e)
  float v_scale;
  int q_bf16;         // query / output dtype for E4M3 KV (16-bit KV: same as the KV dtype)
};

template <int KV, int D>
struct Geom {
  static constexpr int kElt = KV == kKvE4M3 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kRegions = kRowBytes / 128;  // 128-byte column regions per token row
  static constexpr int kColsPerRegion = 128 / kElt;
};

template <int G, int D>
struct MergeSize {
  static constexpr int kBytes = kConsumerWarps * G * D * 4 + kConsumerWarps * G * 8;
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

  __device__ void init(const DecodeParams& p, int seq, int kvh, int lane) {
    grp = lane / kCpr;
    ci = lane % kCpr;
    for (int h = 0; h < G; ++h) {
      const size_t row = (static_cast<size_t>(seq) * p.num_q_heads + kvh * G + h) * D;
      const int d0 = ci * kE;
      load_q(p, row + d0, q[h]);
      for (int e = 0; e < kE; ++e) acc[h][e] = 0.f;
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
  }

  __device__ static void load_q(const DecodeParams& p, size_t idx, float (&dst)[kE]) {
    const bool qbf = (KV == kKvE4M3) ? (p.q_bf16 != 0) : (KV == kKvBF16);
    const uint16_t* qp = static_cast<const uint16_t*>(p.q) + idx;
    for (int e = 0; e < kE; e += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(qp + e);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      for (int k = 0; k < 4; ++k) {
        const float2 f = qbf ? bf16x2_to_float2(w[k]) : f16x2_to_float2(w[k]);
        dst[e + 2 * k] = f.x;
        dst[e + 2 * k + 1] = f.y;
      }
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

  // One 16-token tile: rows r0..r0+15 of the stage, `valid` = bit mask of usable tokens.
  __device__ void tile(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0, uint32_t valid,
                       float score_scale) {
    float s[kIters][G];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int r = it * kGroups + grp;
      const StageRow row = stage_row(r0 + r, p.log2_block, Gm::kRegions, p.region_stride);
      float k[kE];
      load_row(chunk_addr(ks, row, ci, p.region_stride), k);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) dot = fmaf(q[h][e], k[e], dot);
#pragma unroll
        for (int off = 1; off < kCpr; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        s[it][h] = ((valid >> r) & 1u) ? dot * score_scale : -INFINITY;
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
      if (!((valid >> r) & 1u)) continue;
      const StageRow row = stage_row(r0 + r, p.log2_block, Gm::kRegions, p.region_stride);
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

  __device__ void init(const DecodeParams& p, int seq, int kvh, int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    const size_t head0 = static_cast<size_t>(seq) * p.num_q_heads + kvh * G;
    qexp = 1.f;
    if constexpr (kFp8) {
      // Queries go to f16 for the f16 MMA. A power-of-two pre-scale 2^e puts the largest |q|
      // of the group in [2^14, 2^15): exact for every bf16 value in f16's normal range.
      const bool qbf = p.q_bf16 != 0;
      const uint16_t* qp = static_cast<const uint16_t*>(p.q) + head0 * D;
      float amax = 0.f;
      for (int i = lane; i < G * D; i += 32) {
        const uint16_t b = qp[i];
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
            float a = 0.f, b = 0.f;
            if (n < G) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(qp + n * D + d);
              const float2 f = qbf ? bf16x2_to_float2(w) : f16x2_to_float2(w);
              a = f.x * up;
              b = f.y * up;
            }
            qf[nt][j][r] = pack2<false>(a, b);
          }
        }
      }
    } else {
      const uint16_t* qp = static_cast<const uint16_t*>(p.q) + head0 * D;
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        for (int j = 0; j < kK; ++j) {
          for (int r = 0; r < 2; ++r) {
            const int d = 16 * j + 8 * r + 2 * t4;
            qf[nt][j][r] = n < G ? *reinterpret_cast<const uint32_t*>(qp + n * D + d) : 0u;
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

  __device__ void tile(const DecodeParams& p, uint32_t ks, uint32_t vs, int r0, uint32_t valid,
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
        const StageRow row = stage_row(r0 + g + 8 * hi, p.log2_block, Gm::kRegions, p.region_stride);
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
          stage_row(r0 + (lane & 7) + 8 * (i & 1), p.log2_block, Gm::kRegions, p.region_stride);
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
    const bool ok_lo = (valid >> g) & 1u, ok_hi = (valid >> (g + 8)) & 1u;
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
    if (valid != 0xffffu) {
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
        const StageRow ra = stage_row(r0 + 2 * t4 + 8 * pair, p.log2_block, Gm::kRegions, p.region_stride);
        const StageRow rb = stage_row(r0 + 2 * t4 + 8 * pair + 1, p.log2_block, Gm::kRegions, p.region_stride);
        const uint4 x = lds128(chunk_addr(vs, ra, g, p.region_stride));
        const uint4 y = lds128(chunk_addr(vs, rb, g, p.region_stride));
        const uint32_t xa[4] = {x.x, x.y, x.z, x.w};
        const uint32_t ya[4] = {y.x, y.y, y.z, y.w};
        const uint32_t msk = pair ? mask23 : mask01;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t lo = prmt(xa[w], ya[w], 0x5140u);
          const uint32_t hi = prmt(xa[w], ya[w], 0x7362u);
          va[pair][4 * w + 0] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo & 0xffffu)) & msk;
          va[pair][4 * w + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(lo >> 16)) & msk;
          va[pair][4 * w + 2] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi & 0xffffu)) & msk;
          va[pair][4 * w + 3] = e4m3x2_to_f16x2(static_cast<uint16_t>(hi >> 16)) & msk;
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
          stage_row(r0 + (lane & 7) + 8 * (i >> 1), p.log2_block, Gm::kRegions, p.region_stride);
#pragma unroll
      for (int j = 0; j < kK; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(chunk_addr(vs, row, 2 * j + (i & 1), p.region_stride), a0, a1, a2, a3);
        a0 &= mask01;
        a1 &= mask01;
        a2 &= mask23;
        a3 &= mask23;
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

template <int KV, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads)
    pa_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeParams p) {
  using Gm = Geom<KV, D>;
  constexpr bool kMma = G >= 4;
  const bool out_bf16 = KV == kKvE4M3 ? (p.q_bf16 != 0) : (KV == kKvBF16);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(base_ptr + p.ctl_offset);  // full[16], empty[16]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 2 * kMaxStages);
  int* tbl = reinterpret_cast<int*>(bar + 2 * kMaxStages) + 4;
  float* mrg_o = reinterpret_cast<float*>(base_ptr);
  float2* mrg_ml = reinterpret_cast<float2*>(base_ptr + kConsumerWarps * G * D * 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int B = p.block_size;
  const int L = __ldg(p.ctx_lens + seq);
  const size_t out_head0 = static_cast<size_t>(seq) * p.num_q_heads + kvh * G;

  const bool bad_len = L < 0 || L > p.max_ctx || L > p.max_blocks * B;
  if (bad_len || L == 0) {
    if (split == 0) {
      if (bad_len && threadIdx.x == 0) flag_error(p.err, kErrCtxLen);
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) store_out(p.out, out_head0 * D + i, 0.f, out_bf16);
    }
    return;
  }
  const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
  if (split >= nsplit) return;

  const int tok0 = split * p.split_tokens;
  const int tok_end = min(L, tok0 + p.split_tokens);
  const int blk0 = tok0 >> p.log2_block;
  const int nblk = ((tok_end - 1) >> p.log2_block) - blk0 + 1;
  const int st_tokens = max(16, B);
  const int bps = st_tokens >> p.log2_block;
  const int tiles = (tok_end - tok0 + st_tokens - 1) / st_tokens;

  const int32_t* trow = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + blk0;
  for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
    int ph = __ldg(trow + i);
    if (ph < 0 || ph >= p.num_blocks) {
      flag_error(p.err, kErrBlockId);
      ph = -1;
    }
    tbl[i] = ph;
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(bar + s), 1);
      mbar_init(smem_addr(bar + kMaxStages + s), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const uint32_t stage0 = base;  // stage s: K at stage0 + 2*s*stage_bytes, V right after

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      const uint64_t pol = policy_evict_normal();
      const uint32_t tile_bytes = static_cast<uint32_t>(2 * Gm::kRegions * B * 128);
      int issued = 0;
      bool aborted = false;
      for (int t = 0; t < tiles; ++t) {
        const int s = t % p.stages;
        if (t >= p.stages) {
          if (!mbar_wait_bounded(smem_addr(bar + kMaxStages + s), ((t / p.stages) - 1) & 1)) {
            flag_error(p.err, kErrTimeout);
            *abort_flag = 1;
            aborted = true;
            break;
          }
        }
        if (*abort_flag) {
          aborted = true;
          break;
        }
        uint32_t bytes = 0;
        for (int b = 0; b < bps; ++b) {
          const int j = t * bps + b;
          if (j < nblk && tbl[j] >= 0) bytes += tile_bytes;
        }
        const uint32_t full = smem_addr(bar + s);
        mbar_arrive_expect_tx(full, bytes);
        const uint32_t kdst = stage0 + static_cast<uint32_t>(2 * s * p.stage_bytes);
        const uint32_t vdst = kdst + static_cast<uint32_t>(p.stage_bytes);
        for (int b = 0; b < bps; ++b) {
          const int j = t * bps + b;
          if (j >= nblk || tbl[j] < 0) continue;
          const int y = (tbl[j] * p.num_kv_heads + kvh) * B;
          for (int c = 0; c < Gm::kRegions; ++c) {
            const uint32_t off = static_cast<uint32_t>((b * Gm::kRegions + c) * p.region_stride);
            tma_load_2d(kdst + off, &kmap, c * Gm::kColsPerRegion, y, full, pol);
            tma_load_2d(vdst + off, &vmap, c * Gm::kColsPerRegion, y, full, pol);
          }
        }
        issued = t + 1;
      }
      if (aborted) {
        // nothing may still be landing in shared memory when the CTA exits
        for (int t = max(0, issued - p.stages); t < issued; ++t)
          mbar_wait_bounded(smem_addr(bar + (t % p.stages)), (t / p.stages) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int cw = warp - 1;
  Consumer<KV, D, G, kMma> c;
  c.init(p, seq, kvh, lane);
  float score_scale = p.score_scale;
  if constexpr (kMma && KV == kKvE4M3) score_scale *= c.qexp;

  for (int t = cw; t < tiles; t += kConsumerWarps) {
    const int s = t % p.stages;
    if (!mbar_wait_bounded(smem_addr(bar + s), (t / p.stages) & 1)) {
      if (lane == 0) {
        flag_error(p.err, kErrTimeout);
        *abort_flag = 1;
      }
      break;
    }
    const uint32_t ks = stage0 + static_cast<uint32_t>(2 * s * p.stage_bytes);
    const uint32_t vs = ks + static_cast<uint32_t>(p.stage_bytes);
    for (int sub = 0; sub < st_tokens; sub += 16) {
      // validity of the 16 tokens of this tile: inside the context and in a usable block
      const int rt = t * st_tokens + sub + (lane & 15);
      const bool ok = (tok0 + rt < tok_end) && tbl[min(rt >> p.log2_block, nblk - 1)] >= 0;
      const uint32_t valid = __ballot_sync(0xffffffffu, ok && lane < 16) & 0xffffu;
      if (valid == 0) continue;
      c.tile(p, ks, vs, sub, valid, score_scale);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(bar + kMaxStages + s));
    if (*abort_flag) break;
  }

  // merge the consumer warps (the stage ring is reused once every consumer is done with it)
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
  c.publish(mrg_o, mrg_ml, cw, lane);
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");

  const int ctid = threadIdx.x - 32;
  const bool single = nsplit == 1;
  for (int idx = ctid; idx < G * D; idx += kConsumerWarps * 32) {
    const int n = idx / D, d = idx % D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mstar = fmaxf(mstar, mrg_ml[w * G + n].x);
    float num = 0.f, den = 0.f;
    if (mstar != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float2 ml = mrg_ml[w * G + n];
        const float wgt = ex2(ml.x - mstar);
        num = fmaf(wgt, mrg_o[(w * G + n) * D + d], num);
        den = fmaf(wgt, ml.y, den);
      }
    }
    if (single) {
      const float v = den > 0.f ? num / den * p.v_scale : 0.f;
      store_out(p.out, (out_head0 + n) * D + d, v, out_bf16);
    } else {
      const size_t slot = (out_head0 + n) * p.max_splits + split;
      p.part_o[slot * D + d] = num * p.v_scale;
      if (d == 0) p.part_ml[slot] = make_float2(mstar, den);
    }
  }
}

// Combine the split partials of every (sequence, query head) that used more than one split.
// One warp per (sequence, head); lanes own head_dim/32 consecutive outputs.
template <int D>
__global__ void __launch_bounds__(128) pa_reduce_kernel(const __grid_constant__ DecodeParams p,
                                                        int out_bf16) {
  constexpr int kPer = D / 32;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_seqs * p.num_q_heads) return;
  const int seq = gw / p.num_q_heads;
  const int L = __ldg(p.ctx_lens + seq);
  if (L <= 0 || L > p.max_ctx || L > p.max_blocks * p.block_size) return;
  const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
  if (nsplit <= 1) return;
  const size_t slot0 = static_cast<size_t>(gw) * p.max_splits;

  float mstar = -INFINITY;
  for (int i = lane; i < nsplit; i += 32) mstar = fmaxf(mstar, p.part_ml[slot0 + i].x);
  for (int off = 16; off; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));

  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (mstar != -INFINITY) {
    for (int i = 0; i < nsplit; ++i) {
      const float2 ml = p.part_ml[slot0 + i];
      const float wgt = ex2(ml.x - mstar);
      den = fmaf(wgt, ml.y, den);
      const float* src = p.part_o + (slot0 + i) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(wgt, v.x, acc[0]);
        acc[1] = fmaf(wgt, v.y, acc[1]);
        acc[2] = fmaf(wgt, v.z, acc[2]);
        acc[3] = fmaf(wgt, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(wgt, v.x, acc[0]);
        acc[1] = fmaf(wgt, v.y, acc[1]);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e)
    store_out(p.out, static_cast<size_t>(gw) * D + lane * kPer + e, acc[e] * inv, out_bf16 != 0);
}

}  // namespace pa

namespace pa {

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
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  fn<<<grid, kDecodeThreads, smem, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

}  // namespace pa
