// tcgen05_mma_rates.cu - issue and completion rates of tcgen05.mma on one SM (test probe).
//
// One CTA; one thread issues a sequence of kind::f16 MMAs (bf16 operands, fp32 accumulation in
// tensor memory) back to back and commits once at the end (plus the per-group commits a mode
// asks for); the cycles from the first issue to the end of issue and to completion are printed
// per MMA as one JSON line per mode. Operand values do not matter (shared memory holds a
// constant pattern). The modes are the shapes and orders an attention kernel uses:
//   0  M128 N64  K16, A and B K-major in shared memory (an S tile of 64 keys)
//   1  M128 N128 K16, A and B K-major in shared memory
//   2  M128 N128 K16, A from tensor memory, B MN-major in shared memory (a PV step)
//   3  M128 N256 K16, A and B K-major in shared memory
//   4  one query tile: S (8 MMAs, N64, shared-memory operands) then PV (4 MMAs, N128, B MN-major,
//      another accumulator), alternating: accumulator, N and B major all change between groups
//   5  attention order over 64-key tiles for two query tiles: S_0, S_1 (8 MMAs each, N64), then
//      PV_0, PV_1 (4 MMAs each, N128, P from shared memory); each S_x at a fixed column
//   6  mode 5 with S_x double-buffered at columns c and c + 64 (one 128-column group), the
//      buffer alternating tile by tile
//   7  mode 6 with one commit after the S pair and one after the PV pair
// Modes 0-7 build each MMA's descriptors in the issue loop; modes 8-10 build them before the
// loop and unroll each group, so that only the MMAs (and commits) are issued:
//   8  mode 6's sequence (S double-buffered, as in the prefill kernel)
//   9  mode 4's sequence with one commit after each group
//  10  mode 4's sequence with two commits after each group
// Every wait is bounded; a timeout is reported as status 1.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

namespace {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// shared-memory matrix descriptor, 128-byte swizzle, version 1
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3fffu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, B major bit, N, M
__device__ __forceinline__ uint32_t idesc(int m, int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, 1, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d), "l"(a), "l"(b), "r"(id) : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, 1, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
      ::"r"(d), "r"(a), "l"(b), "r"(id) : "memory");
}

__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
    if ((i & 255u) == 0 && clock64() - t0 > 2000000000ll) return false;
  }
}

constexpr int kMmas = 672;  // a multiple of 12 and of 24 (whole groups in modes 4-10)

template <int MODE>
__global__ void rates(long long* out, int* status) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t done, groups;
  __shared__ uint32_t tbase;
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&done)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&groups)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(saddr(&tbase)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x3c003c00u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t t = tbase;
  const uint32_t a = saddr(sm), b = a + 32768;  // A: 32 KB, B: 32 KB
  if (threadIdx.x == 0 && MODE >= 8) {
    uint64_t dq[4], dk[4], dp[4], dv[4];  // S: Q and K steps; PV: P and V steps
    for (int k = 0; k < 4; ++k) {
      dq[k] = desc(a + k * 32, 16, 1024);
      dk[k] = desc(b + k * 32, 16, 1024);
      dp[k] = desc(a + 16384 + k * 32, 16, 1024);
      dv[k] = desc(b + k * 2048, 8192, 1024);
    }
    const uint32_t idS = idesc(128, 64, 0), idO = idesc(128, 128, 1);
    const long long c0 = clock64();
    if (MODE == 8) {
      for (int tile = 0; tile < kMmas / 24; ++tile) {
        const uint32_t sbuf = 64u * (tile & 1);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int k = 0; k < 8; ++k) mma_ss(t + 256 + 128 * x + sbuf, dq[k & 3], dk[k & 3], idS);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(t + 128 * x, dp[k], dv[k], idO);
      }
    } else {
      for (int tile = 0; tile < kMmas / 12; ++tile) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_ss(t + 256, dq[k & 3], dk[k & 3], idS);
        commit(saddr(&groups));
        if (MODE == 10) commit(saddr(&groups));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_ss(t, dp[k], dv[k], idO);
        commit(saddr(&groups));
        if (MODE == 10) commit(saddr(&groups));
      }
    }
    const long long c1 = clock64();
    commit(saddr(&done));
    const bool ok = wait_bounded(saddr(&done), 0);
    const long long c2 = clock64();
    out[0] = c1 - c0;
    out[1] = c2 - c0;
    if (!ok) *status = 1;
  } else if (threadIdx.x == 0) {
    const long long c0 = clock64();
    for (int i = 0; i < kMmas; ++i) {
      const int k = i & 3;
      if (MODE == 0) {
        mma_ss(t + 256, desc(a + k * 32, 16, 1024), desc(b + k * 32, 16, 1024), idesc(128, 64, 0));
      } else if (MODE == 1) {
        mma_ss(t + 256, desc(a + k * 32, 16, 1024), desc(b + k * 32, 16, 1024), idesc(128, 128, 0));
      } else if (MODE == 2) {
        mma_ts(t, t + 256 + k * 8, desc(b + k * 2048, 8192, 1024), idesc(128, 128, 1));
      } else if (MODE == 3) {
        mma_ss(t + 256, desc(a + k * 32, 16, 1024), desc(b + k * 32, 16, 1024), idesc(128, 256, 0));
      } else if (MODE == 4) {
        if (i % 12 < 8)
          mma_ss(t + 256, desc(a + k * 32, 16, 1024), desc(b + k * 32, 16, 1024), idesc(128, 64, 0));
        else
          mma_ss(t, desc(a + 16384 + k * 32, 16, 1024), desc(b + k * 2048, 8192, 1024),
                 idesc(128, 128, 1));
      } else {
        const int ph = i % 24, tile = i / 24;
        const uint32_t sbuf = MODE == 5 ? 0u : 64u * (tile & 1);
        if (ph < 16)
          mma_ss(t + 256 + (ph >= 8 ? 128u : 0u) + sbuf, desc(a + k * 32, 16, 1024),
                 desc(b + k * 32, 16, 1024), idesc(128, 64, 0));
        else
          mma_ss(t + (ph >= 20 ? 128u : 0u), desc(a + 16384 + k * 32, 16, 1024),
                 desc(b + k * 2048, 8192, 1024), idesc(128, 128, 1));
        if (MODE == 7 && (ph == 15 || ph == 23)) commit(saddr(&groups));
      }
    }
    const long long c1 = clock64();
    commit(saddr(&done));
    const bool ok = wait_bounded(saddr(&done), 0);
    const long long c2 = clock64();
    out[0] = c1 - c0;
    out[1] = c2 - c0;
    if (!ok) *status = 1;
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(t));
}

template <int MODE>
cudaError_t launch(long long* d, int* st) {
  const int smem = 65536 + 1024;
  cudaError_t e = cudaFuncSetAttribute(rates<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  rates<MODE><<<1, 128, smem>>>(d, st);
  return cudaGetLastError();
}

}  // namespace

int main() {
  long long* d = nullptr;
  int* st = nullptr;
  if (cudaMalloc(&d, 16) != cudaSuccess || cudaMalloc(&st, 4) != cudaSuccess) return 2;
  constexpr int kModes = 11;
  const char* names[kModes] = {"N64 smem A", "N128 smem A", "N128 tmem A (PV)", "N256 smem A",
                               "S / PV alternating, one query tile", "attention, S at fixed columns",
                               "attention, S double-buffered in one 128-column group",
                               "attention, S double-buffered, commits",
                               "attention, S double-buffered (mode 6), precomputed",
                               "one query tile, precomputed, 1 commit per group",
                               "one query tile, precomputed, 2 commits per group"};
  // flops per MMA averaged over the mode's sequence
  const double f64 = 128.0 * 64 * 16 * 2, f128 = 128.0 * 128 * 16 * 2;
  const double mix = (16 * f64 + 8 * f128) / 24;
  const double flops[kModes] = {f64, f128, f128, 2 * f128, mix, mix, mix, mix, mix, mix, mix};
  for (int mode = 0; mode < kModes; ++mode) {
    long long h[2] = {0, 0};
    int hs = 0;
    for (int rep = 0; rep < 3; ++rep) {  // the last of three runs is reported
      cudaMemset(st, 0, 4);
      cudaError_t e = cudaSuccess;
      switch (mode) {
        case 0: e = launch<0>(d, st); break;
        case 1: e = launch<1>(d, st); break;
        case 2: e = launch<2>(d, st); break;
        case 3: e = launch<3>(d, st); break;
        case 4: e = launch<4>(d, st); break;
        case 5: e = launch<5>(d, st); break;
        case 6: e = launch<6>(d, st); break;
        case 7: e = launch<7>(d, st); break;
        case 8: e = launch<8>(d, st); break;
        case 9: e = launch<9>(d, st); break;
        default: e = launch<10>(d, st); break;
      }
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) {
        printf("{\"mode\": %d, \"error\": \"%s\"}\n", mode, cudaGetErrorString(e));
        return 1;
      }
      cudaMemcpy(h, d, 16, cudaMemcpyDeviceToHost);
      cudaMemcpy(&hs, st, 4, cudaMemcpyDeviceToHost);
    }
    printf("{\"mode\": %d, \"name\": \"%s\", \"issue_cycles_per_mma\": %.1f, "
           "\"cycles_per_mma\": %.1f, \"flop_per_cycle\": %.0f, \"status\": %d}\n",
           mode, names[mode], h[0] / static_cast<double>(kMmas), h[1] / static_cast<double>(kMmas),
           flops[mode] * kMmas / static_cast<double>(h[1]), hs);
  }
  return 0;
}
