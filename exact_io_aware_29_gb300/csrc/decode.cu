// Decoding from a paged KV cache: one new query per (sequence, head) attends
// to the sequence's L cached keys, which live in fixed-size pages of a shared
// pool and are found through a per-sequence block table ("FlashAttention
// 完整解析", §7.2-7.4: PageAttention block tables; the online softmax of
// "FlashAttention算法详解", §Online Softmax).
//
// With one query row there is no matrix product to feed the tensor cores: the
// step reads every cached K and V byte once and does ~1 flop per byte, so HBM
// bandwidth is the bound. The design follows from that:
//   * one warp streams 64-key K and V tiles with TMA (the pool is viewed as a
//     packed [num_blocks * block_size, H, d] tensor; a tile never crosses a
//     page because block_size is a multiple of 64) through a ring of stages
//     deep enough to keep ~190 KB in flight per SM;
//   * eight consumer warps split each tile: a group of d/8 lanes owns one key
//     at a time (16 bytes of the row per lane), reduces q . k with shuffles,
//     and keeps an exact fp32 online softmax (m, l, o) per group;
//   * a sequence's keys are split across CTAs (chunks of whole tiles) so that
//     short batches still fill the GPU; groups are merged in shared memory,
//     splits by a small combine kernel in fixed split order (deterministic).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {

template <int D>
struct DecCfg {
  static constexpr int TK = 64;                      // keys per tile (TMA box height)
  static constexpr int BOXES = D / 64;               // 64-column boxes per row
  static constexpr int BOX_BYTES = TK * 128;         // 64 rows x 64 bf16, 128B-swizzled
  static constexpr int TILE_BYTES = BOXES * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile, then V tile
  static constexpr int STAGES = D == 128 ? 6 : 10;
  static constexpr int CWARPS = 8;                   // consumer warps
  static constexpr int THREADS = 32 * (CWARPS + 1);  // + the TMA warp
  static constexpr int LPK = D / 8;                  // lanes per key (16 bytes each)
  static constexpr int GROUPS = CWARPS * 32 / LPK;   // keys in flight per CTA step
  static constexpr int KPG = TK / GROUPS;            // keys per group per tile
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 2 * STAGES * 8 + 16 + 1024;  // + alignment slack
  static_assert(KPG * GROUPS == TK, "tile split");
  static_assert(GROUPS * (D + 2) * 4 <= OFF_BAR, "merge buffer fits in the stages");
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const DecodeArgs a) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::STAGES);

  const int BH = a.B * a.H;
  const int split = blockIdx.x / BH;  // split-major: first splits of every head run first
  const int bh = blockIdx.x - split * BH;
  const int b = bh / a.H, h = bh - b * a.H;
  int L = a.seq_lens[b];
  L = L < 0 ? 0 : (L > a.max_seq_len ? a.max_seq_len : L);
  const int nsplit_b = L == 0 ? 1 : (L + a.chunk - 1) / a.chunk;
  if (split >= nsplit_b) return;  // the whole CTA: nothing to do for this split
  const int c0 = split * a.chunk;
  const int c1 = min(L, c0 + a.chunk);
  const int ntiles = c1 > c0 ? (c1 - c0 + C::TK - 1) / C::TK : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::CWARPS) {
    // ------------------------------------------------------------ TMA warp
    if (lane == 0 && !g_test_drop_loads) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % C::STAGES, use = t / C::STAGES;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag)) break;
        const int key = c0 + t * C::TK;
        const int page = key / a.block_size;
        const int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks + page];
        // Out-of-range block ids read as zeros (TMA fills outside the pool).
        const int row = (phys < 0 || phys >= a.num_blocks) ? -C::TK : phys * a.block_size + (key - page * a.block_size);
        uint8_t* st = smem + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
        for (int c = 0; c < C::BOXES; ++c) {
          tma_load_3d(st + c * C::BOX_BYTES, &tmK, &full[s], c * 64, h, row);
          tma_load_3d(st + C::TILE_BYTES + c * C::BOX_BYTES, &tmV, &full[s], c * 64, h, row);
        }
        ++issued;
      }
      // Do not leave with copies in flight (matters only after an abort, when
      // the consumers stopped waiting; every issued copy lands).
      for (int t = max(0, issued - C::STAGES); t < issued; ++t) mbar_wait_drain(&full[t % C::STAGES], (t / C::STAGES) & 1);
    }
  } else {
    // ------------------------------------------------------ consumer warps
    const int grp = (warp * 32 + lane) / C::LPK;  // 0..GROUPS-1
    const int seg = lane % C::LPK;                // 16-byte segment of the row
    const int box = seg >> 3, ch = seg & 7;       // 64-column box, 16-byte chunk in it
    float q[8];
    {
      const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                       static_cast<size_t>(bh) * D + seg * 8);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q[2 * i] = bf16_lo(ww[i]) * a.scale_log2;  // logits in base-2 units
        q[2 * i + 1] = bf16_hi(ww[i]) * a.scale_log2;
      }
    }
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % C::STAGES;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (t / C::STAGES) & 1, abort_flag));
      if (!ok) break;
      const uint8_t* Kt = smem + s * C::STAGE_BYTES + box * C::BOX_BYTES;
      const uint8_t* Vt = Kt + C::TILE_BYTES;
      const int kbase = c0 + t * C::TK;
      float sc[C::KPG];
#pragma unroll
      for (int i = 0; i < C::KPG; ++i) {
        const int r = grp + i * C::GROUPS;  // row of the tile
        const uint4 w = *reinterpret_cast<const uint4*>(Kt + r * 128 + ((ch ^ (r & 7)) << 4));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        float dot = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          dot = fmaf(q[2 * k2], bf16_lo(ww[k2]), dot);
          dot = fmaf(q[2 * k2 + 1], bf16_hi(ww[k2]), dot);
        }
#pragma unroll
        for (int off = C::LPK / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        sc[i] = (kbase + r < c1) ? dot : -INFINITY;
      }
      float mx = m;
#pragma unroll
      for (int i = 0; i < C::KPG; ++i) mx = fmaxf(mx, sc[i]);
      if (mx > -INFINITY) {
        const float alpha = ex2(m - mx);  // 0 while nothing was seen (m = -inf)
        l *= alpha;
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] *= alpha;
#pragma unroll
        for (int i = 0; i < C::KPG; ++i) {
          const int r = grp + i * C::GROUPS;
          const float p = ex2(sc[i] - mx);
          l += p;
          const uint4 w = *reinterpret_cast<const uint4*>(Vt + r * 128 + ((ch ^ (r & 7)) << 4));
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            o[2 * k2] = fmaf(p, bf16_lo(ww[k2]), o[2 * k2]);
            o[2 * k2 + 1] = fmaf(p, bf16_hi(ww[k2]), o[2 * k2 + 1]);
          }
        }
        m = mx;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // Merge the groups: every consumer is past its last tile, so the stage
    // memory (all copies landed) is free for the partial results.
    named_bar_sync(1, C::CWARPS * 32);
    float* red_o = reinterpret_cast<float*>(smem);       // [GROUPS][D]
    float* red_ml = red_o + C::GROUPS * D;               // [GROUPS][2]
#pragma unroll
    for (int j = 0; j < 8; ++j) red_o[grp * D + seg * 8 + j] = o[j];
    if (seg == 0) {
      red_ml[2 * grp] = m;
      red_ml[2 * grp + 1] = l;
    }
    named_bar_sync(1, C::CWARPS * 32);
    const int tid = threadIdx.x;
    if (tid < D) {
      float M = -INFINITY;
      for (int g = 0; g < C::GROUPS; ++g) M = fmaxf(M, red_ml[2 * g]);
      float lsum = 0.f, acc = 0.f;
      if (M > -INFINITY) {
        for (int g = 0; g < C::GROUPS; ++g) {
          const float mg = red_ml[2 * g];
          if (mg == -INFINITY) continue;
          const float f = ex2(mg - M);
          lsum = fmaf(red_ml[2 * g + 1], f, lsum);
          acc = fmaf(red_o[g * D + tid], f, acc);
        }
      }
      if (nsplit_b == 1) {
        const float outv = lsum > 0.f ? acc / lsum : 0.f;
        static_cast<__nv_bfloat16*>(a.o)[static_cast<size_t>(bh) * D + tid] = __float2bfloat16_rn(outv);
        if (tid == 0) a.lse[bh] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
      } else {
        const size_t p = static_cast<size_t>(bh) * a.nsplit + split;
        a.part_o[p * D + tid] = acc;
        if (tid == 0) {
          a.part_ml[2 * p] = M;
          a.part_ml[2 * p + 1] = lsum;
        }
      }
    }
  }
}

// Merges the splits of each (sequence, head) in split order.
template <int D>
__global__ void __launch_bounds__(D) fa_decode_combine_kernel(const DecodeArgs a) {
  const int bh = blockIdx.x;
  const int b = bh / a.H;
  int L = a.seq_lens[b];
  L = L < 0 ? 0 : (L > a.max_seq_len ? a.max_seq_len : L);
  const int ns = L == 0 ? 1 : (L + a.chunk - 1) / a.chunk;
  if (ns <= 1) return;  // written by the decode kernel
  const size_t p0 = static_cast<size_t>(bh) * a.nsplit;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, a.part_ml[2 * (p0 + s)]);
  float lsum = 0.f, acc = 0.f;
  if (M > -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float ms = a.part_ml[2 * (p0 + s)];
      if (ms == -INFINITY) continue;
      const float f = ex2(ms - M);
      lsum = fmaf(a.part_ml[2 * (p0 + s) + 1], f, lsum);
      acc = fmaf(a.part_o[(p0 + s) * D + threadIdx.x], f, acc);
    }
  }
  static_cast<__nv_bfloat16*>(a.o)[static_cast<size_t>(bh) * D + threadIdx.x] =
      __float2bfloat16_rn(lsum > 0.f ? acc / lsum : 0.f);
  if (threadIdx.x == 0) a.lse[bh] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
}

template <int D>
static cudaError_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                   cudaStream_t stream, const LaunchMarks* marks) {
  using C = DecCfg<D>;
  auto kern = fa_decode_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(a.B) * a.H * a.nsplit;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  mark(marks, true, 0, stream);
  kern<<<static_cast<unsigned>(blocks), C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, a);
  mark(marks, false, 0, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.nsplit == 1) return e;
  mark(marks, true, 1, stream);
  fa_decode_combine_kernel<D><<<static_cast<unsigned>(a.B * a.H), D, 0, stream>>>(a);
  mark(marks, false, 1, stream);
  return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t stream,
                          const LaunchMarks* m) {
  return a.D == 64 ? launch_decode_t<64>(tk, tv, a, stream, m) : launch_decode_t<128>(tk, tv, a, stream, m);
}

cudaError_t set_decode_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_decode_status() { return take_status_here(); }

}  // namespace fa
