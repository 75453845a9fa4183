// Backward pass of exact attention on sm_103a.
//
// Gradients of L = sum(O * dO) by the formulas of "FlashAttention算法详解：从
// IO瓶颈到Triton实现", §Backward为什么更复杂: dV = P^T dO, dP = dO V^T,
// dS = P o (dP - rowsum(dP o P)), dQ = scale * dS K, dK = scale * dS^T Q, with P
// recomputed block by block from the saved row LSE (P_ij = exp(S_ij - LSE_i))
// instead of being stored (youngju.dev flash_attention.zh §7.2). The row term
// rowsum(dP o P) equals rowsum(dO o O) because O = P V, so it is formed once per
// query row from dO and O by a small pre-pass.
//
// Kernels:
//   bwd_pre      delta = rowsum(dO o O), nlse2 = -LSE * log2(e) (-inf for
//                rows with no visible key and for padding rows), dq_acc = 0.
//   bwd_main     persistent, one CTA per SM; a work item is (b, h, 128-key
//                block j), with a loop over the 128-query blocks i that see
//                block j (causal: i >= j), all in TMEM/SMEM:
//                  S^T  = K_j Q_i^T             (tcgen05, TMEM region R[i%2])
//                  P^T  = 2^(S^T * scale*log2e + nlse2_i)  (bf16, back into R[i%2])
//                  dP^T = V_j dO_i^T            (R[i%2] again, after dV read P^T)
//                  dV  += P^T dO_i              (A = P^T from TMEM)
//                  dS^T = P^T o (dP^T - delta_i) (bf16, to TMEM over dP^T and
//                                                to shared memory)
//                  dK  += dS^T Q_i              (A = dS^T from TMEM)
//                  dQ_i = dS K_j                (A = dS^T in shared memory read as
//                                                MN-major; into R[i%2])
//                and a warpgroup stages dQ_i in shared memory and adds it to
//                the fp32 accumulator with bulk asynchronous reductions.
//                dK (times scale) and dV leave as bf16.
//   bwd_dq       dQ = scale * dq_acc, bf16.
// Warp roles of bwd_main (16 warps): warp 0 TMA producer (it also claims the
// work items), warp 1 tcgen05 issuer of S^T, dV and dP^T, warp 14 issuer of dK
// and dQ, warps 2-5 and 6-9 one key row per thread for query columns 0-63 and
// 64-127 (P^T, dS^T, then half of the dK/dV epilogue each), warps 10-13 one
// query row per thread (dQ_i readout and reduction), warp 15 the zero dK/dV
// rows of key blocks no query sees. Any four consecutive warps cover the four
// TMEM lane quarters (warp w reads lanes 32*(w%4)..+31). In the deterministic
// order warp 1 issues every product and warp 14 issues the dQ reductions in a
// fixed order across CTAs (see the dQ reduction issuer).
//
// dQ accumulator layout (private to the library): per (b*h, 128-query block,
// 64-column half) a 32 KB tile stored as [16 float4 column groups][128 rows],
// so the staging writes in shared memory are bank-conflict free and each
// 32-column quarter (16 KB) is one contiguous bulk reduction.
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;  // queries per block
  static constexpr int BN = 128;  // keys per CTA
  static constexpr int CHUNKS = D / 64;
  static constexpr int HALVES = D / 64;     // 64-column halves of a dQ tile
  static constexpr int TILE = 128 * D * 2;  // one [128 x D] bf16 tile
  static constexpr int SUB = 128 * 128;     // one [128 rows x 64 cols] swizzled chunk
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;    // 2 slots
  static constexpr int OFF_DO = 4 * TILE;   // 1 slot
  static constexpr int OFF_DS = 5 * TILE;   // dS^T [128 keys x 128 queries] bf16
  static constexpr int OFF_STAGE = OFF_DS + 2 * SUB;   // dQ staging: two 16 KB buffers, 128 rows x 32 fp32 each
  static constexpr int OFF_VEC = OFF_STAGE + 32768;    // 2 slots x (nlse2[128], delta[128]) fp32
  static constexpr int OFF_BAR = OFF_VEC + 2 * 1024;
  static constexpr int NUM_BARS = 28;
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16;  // + TMEM address, abort flag, item ring
  static constexpr int THREADS = 512;
  static constexpr uint32_t TMEM_COLS = 512;
};

// ---------------------------------------------------------------------------
// Pre-pass: delta, nlse2, zeroed dQ accumulator. Rows are padded per head to a
// multiple of 128 (Npad) so every 128-row block is whole.
// ---------------------------------------------------------------------------
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdArgs a, int Npad) {
  constexpr int TPR = D / 8;  // threads per row, 8 columns each
  const int N = a.s.N;
  const size_t rows = static_cast<size_t>(a.s.B) * a.s.H * Npad;
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t row = tid / TPR;
  const int g = static_cast<int>(tid % TPR);
  const bool in_range = row < rows;
  // Workspace state first: it depends on nothing the forward writes, so with
  // a programmatic launch it overlaps the forward's last CTAs. Counters of the
  // deterministic order (one per 128-row block) and the ticket, then the
  // accumulator, which has exactly D floats per padded row.
  if (tid < rows / 128) a.dq_turn[tid] = 0u;
  if (tid == 0) *a.ticket = 0u;
  if (in_range) {
    float4* z = reinterpret_cast<float4*>(a.dq_acc + row * D + g * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();  // O and LSE come from the forward
  const size_t bh = in_range ? row / Npad : 0;
  const int n = in_range ? static_cast<int>(row % Npad) : 0;
  const SeqView sv = seq_view<VARLEN>(a.pk, a.kv_lens, static_cast<int>(bh / a.s.H), N);
  const bool real = in_range && n < sv.Lq;
  float acc = 0.f;
  if (real) {
    const size_t off = q_row<VARLEN>(a.pk, a.s, sv, static_cast<int>(bh), n) * D + g * 8;
    const uint4 o4 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o) + off);
    const uint4 d4 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.dO) + off);
    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
    const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(dw[i] << 16), acc);
      acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(dw[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (!in_range) return;
  if (g == 0) {
    a.delta[row] = acc;
    float nl2 = -INFINITY;  // 2^(x + nl2) = 0: the row contributes nothing
    if (real) {
      const float l = a.lse[lse_index<VARLEN>(a.pk, a.s, sv, static_cast<int>(bh), n)];
      if (l > -INFINITY) nl2 = -l * kLog2e;
    }
    a.lse2[row] = nl2;
  }
}

// ---------------------------------------------------------------------------
// dQ = scale * dq_acc -> bf16. One block per 32 KB accumulator tile (128 rows
// x 64 columns): contiguous float4 reads (consecutive threads, consecutive
// rows of one column group), converted into a shared-memory copy of the tile
// in row order, then written as whole 128-byte row segments (eight threads
// per row) instead of 16 bytes in each of 32 rows per warp instruction.
// ---------------------------------------------------------------------------
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdArgs a, int Npad) {
  constexpr int HALVES = D / 64;
  constexpr int LD = 68;  // bf16 per shared row: 34 words, so the 8-byte writes of 32 rows spread over all banks
  __shared__ __align__(16) uint16_t tile[128 * LD];
  const int nqb = Npad / 128;
  griddep_wait();  // the accumulator is complete once the main kernel has finished
  // Last tiles first: the main kernel finishes with the last group of heads,
  // whose accumulator tiles are still in L2 when this kernel starts (C4:
  // 33.0 -> 31.2 us).
  const size_t t = gridDim.x - 1 - blockIdx.x;  // (bh * nqb + qb) * HALVES + hh
  const int hh = static_cast<int>(t % HALVES);
  const int qb = static_cast<int>((t / HALVES) % nqb);
  const int bh = static_cast<int>(t / HALVES / nqb);
  const SeqView sv = seq_view<VARLEN>(a.pk, a.kv_lens, bh / a.s.H, a.s.N);
  const int rows = min(128, sv.Lq - qb * 128);
  if (rows <= 0) return;
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc) + t * (16 * 128);
  const float s = a.s.scale;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int e = threadIdx.x + 256 * k;  // column group e / 128, row e % 128
    const float4 x = src[e];
    uint2 w;
    w.x = pack_bf16x2(x.x * s, x.y * s);
    w.y = pack_bf16x2(x.z * s, x.w * s);
    *reinterpret_cast<uint2*>(&tile[(e & 127) * LD + (e >> 7) * 4]) = w;
  }
  __syncthreads();
  uint16_t* dq = static_cast<uint16_t*>(a.dq);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = threadIdx.x + 256 * k;
    const int r = e >> 3, part = e & 7;  // 8 columns per thread
    if (r < rows) {
      const uint2 lo = *reinterpret_cast<const uint2*>(&tile[r * LD + part * 8]);
      const uint2 hi = *reinterpret_cast<const uint2*>(&tile[r * LD + part * 8 + 4]);
      *reinterpret_cast<uint4*>(dq + q_row<VARLEN>(a.pk, a.s, sv, bh, qb * 128 + r) * D + hh * 64 + part * 8) =
          make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  }
}

// ---------------------------------------------------------------------------
// Main kernel
// ---------------------------------------------------------------------------
// One work item: key block j of flattened head bh, with the query blocks that
// see it. Items are numbered in the grid order described below.
struct BwdWork {
  int bh, j, key0, i_lo, n_iter;
  SeqView sv;
};

template <int D, bool CAUSAL, bool VARLEN, bool DET>
__device__ __forceinline__ BwdWork bwd_work(const BwdArgs& args, int item) {
  using C = BwdCfg<D>;
  const AttnShape& sh = args.s;
  const int nkb = (sh.Nk + C::BN - 1) / C::BN;
  // Groups of heads run together, so their Q, dO and dQ accumulators stay in
  // L2 (the launch sizes a group to the L2). Default order: inside a group the
  // key blocks go heaviest first (causal: block j sees nkb - j query blocks)
  // across the group's heads; deterministic order: lightest first, see the
  // dQ reduction issuer.
  const int BH = sh.B * sh.H;
  const int G = min(BH, max(1, args.heads_per_group));
  const int group = item / (G * nkb);
  const int gsize = min(G, BH - group * G);
  const int r_in = item - group * G * nkb;
  BwdWork w;
  w.j = DET ? nkb - 1 - r_in / gsize : r_in / gsize;
  w.bh = group * G + r_in % gsize;
  w.sv = seq_view<VARLEN>(args.pk, args.kv_lens, w.bh / sh.H, sh.N);
  w.key0 = w.j * C::BN;
  // Query r sees key c iff c <= r + shift (causal): the first query block that
  // sees key block j starts at row key0 - shift.
  // (Fixed layout: shift 0, every sequence nkb query blocks long.)
  w.i_lo = CAUSAL ? (VARLEN ? max(0, w.key0 - w.sv.shift) / C::BM : w.j) : 0;
  const int nq = VARLEN ? (w.sv.Lq + C::BM - 1) / C::BM : nkb;  // query blocks of this sequence
  w.n_iter = (w.key0 >= w.sv.Lk) ? 0 : (VARLEN ? max(0, nq - w.i_lo) : nkb - w.i_lo);
  return w;
}

// Persistent: one CTA per SM takes work items from a global ticket counter
// until none is left. Every mbarrier is used either once per block pair (its
// phase is the pair's index p, counted over all of this CTA's items) or once
// per item (phase = item index); TMEM, the barriers and the operand
// descriptors are set up once, and while one item drains (last dQ reductions,
// dK/dV epilogue) the next one's K, V, Q and dO already load and its first
// S^T runs.
template <int D, bool CAUSAL, bool VARLEN, bool DET>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdArgs args) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The swizzled tiles need a 1024-byte aligned base; the layout has no slack.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicExch(&g_fa_status, kStatusTimeout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars + 0;    // per item
  uint64_t* q_full = bars + 1;    // [2] Q_i tile + nlse2/delta vectors
  uint64_t* q_empty = bars + 3;   // [2]
  uint64_t* do_full = bars + 5;
  uint64_t* do_empty = bars + 6;
  uint64_t* s_full = bars + 7;
  uint64_t* dp_full = bars + 8;
  uint64_t* p_ready = bars + 9;    // 256 arrivals
  uint64_t* ds_ready = bars + 10;  // 256 arrivals
  uint64_t* dq_full = bars + 11;
  uint64_t* dq_empty = bars + 12;  // 128 arrivals
  uint64_t* mma_done = bars + 13;  // per item: every product of the item has completed
  // Deterministic order: staging buffer b (of two) filled (128 arrivals) and
  // read out by its reduction.
  uint64_t* stage_full[2] = {bars + 14, bars + 24};
  uint64_t* stage_free[2] = {bars + 15, bars + 25};
  uint64_t* v_full = bars + 16;      // per item
  uint64_t* item_full = bars + 17;   // [2] item ring
  uint64_t* item_empty = bars + 19;  // [2] one arrival per consuming warp
  uint64_t* ds_free = bars + 21;     // dQ_p has read dS^T_p from shared memory
  uint64_t* epi_full = bars + 22;    // dK/dV epilogue: staged (256 arrivals)
  uint64_t* epi_empty = bars + 23;   // dK/dV epilogue: copied out (256 arrivals)
  uint64_t* fin = bars + 26;         // [2] per issuing thread: all its MMAs have completed (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  constexpr int kItemConsumers = 14;  // warps 1 and 14 (one thread each), 2-9, 10-13

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int nkb = (sh.Nk + C::BN - 1) / C::BN;  // key blocks per head
  const int nqb = (N + C::BM - 1) / C::BM;       // query blocks of the padded workspace
  const int Npad = nqb * C::BM;
  const int n_items = sh.B * sh.H * nkb;
  constexpr bool packed = VARLEN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NUM_BARS; ++i) mbar_init(&bars[i], 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_empty, 128);
    mbar_init(mma_done, DET ? 1 : 2);  // one commit per issuing thread
    if (DET) {
      mbar_init(stage_full[0], 128);
      mbar_init(stage_full[1], 128);
    }
    mbar_init(&item_empty[0], kItemConsumers);
    mbar_init(&item_empty[1], kItemConsumers);
    mbar_init(epi_full, 256);
    mbar_init(epi_empty, 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tR0 = tmem, tR1 = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + D;
  // Set-up above overlaps the pre-pass's last CTAs (programmatic launch);
  // everything below reads what the pre-pass writes (ticket, delta, nlse2,
  // zeroed accumulator). The dQ conversion may then launch and wait in turn.
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();

  // Item ci of this CTA from the ring, or -1 when there is none (or the wait
  // ran out). take_item: one thread; take_item_warp: a whole converged warp,
  // lane 0 waits and reads for it.
  auto take_item = [&](int ci) -> int {
    const int rs = ci & 1;
    if (!mbar_wait(&item_full[rs], (ci >> 1) & 1, abort_flag)) return -1;
    const int w = item_ring[rs];
    mbar_arrive(&item_empty[rs]);
    return w;
  };
  auto take_item_warp = [&](int ci) -> int {
    const int w = lane == 0 ? take_item(ci) : -1;
    return __shfl_sync(0xffffffffu, w, 0);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && !g_test_drop_loads) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      int ci = 0;  // items published
      int pc = 0;  // block pairs loaded, over all items
      // K, V, Q-slot and dO loads issued, set where a wait gives up in the
      // middle of an item (else derived from ci and pc after the loop).
      int kn = -1, vn = 0, qn = 0, dn = 0;
      bool ok = true;
      for (;; ++ci) {
        // Claim the next item that has work (warp 15 writes the zero
        // gradients of key blocks that no query sees).
        int w = -1;
        BwdWork wk;
        for (;;) {
          const int t = static_cast<int>(atomicAdd(args.ticket, 1u));
          if (t >= n_items) break;
          wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, t);
          if (wk.n_iter > 0) {
            w = t;
            break;
          }
        }
        const int rs = ci & 1;
        if (ci >= 2 && !(ok = mbar_wait(&item_empty[rs], ((ci - 2) >> 1) & 1, abort_flag))) break;
        item_ring[rs] = w;
        mbar_arrive(&item_full[rs]);
        if (w < 0) break;
        // K and V trade buffers from one item to the next: this item's K goes
        // where the previous item's V was (free once the previous item's last
        // dP^T has completed: do_empty of its last pair), its V where the
        // previous K was (free once every product of the previous item has
        // completed: mma_done). So the first S^T of this item can run before
        // the previous item's last dK and dQ are done.
        const int kbuf = (ci & 1) ? C::OFF_V : C::OFF_K, vbuf = (ci & 1) ? C::OFF_K : C::OFF_V;
        if (pc > 0 && !(ok = mbar_wait(do_empty, (pc - 1) & 1, abort_flag))) break;
        // K and Q_0 first: S^T_0 needs only them; V is first read by dP^T_0.
        const int head = wk.bh % sh.H;
        const int ky = packed ? head : wk.key0, kz = packed ? wk.sv.k_start + wk.key0 : wk.bh;
        mbar_arrive_expect_tx(k_full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) tma_load_3d(smem + kbuf + c * C::SUB, &tmK, k_full, c * 64, ky, kz);
        for (int it = 0; it < wk.n_iter; ++it) {
          const int p = pc + it;
          const int slot = p & 1, use = p >> 1;
          const int qb = wk.i_lo + it;
          const int qy = packed ? head : qb * C::BM, qz = packed ? wk.sv.q_start + qb * C::BM : wk.bh;
          if (use > 0 && !(ok = mbar_wait(&q_empty[slot], (use - 1) & 1, abort_flag))) {
            kn = ci + 1, vn = ci + (it > 0 ? 1 : 0), qn = p, dn = p;
            break;
          }
          mbar_arrive_expect_tx(&q_full[slot], C::TILE + 1024);
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_3d(smem + C::OFF_Q + slot * C::TILE + c * C::SUB, &tmQ, &q_full[slot], c * 64, qy, qz);
          const size_t voff = static_cast<size_t>(wk.bh) * Npad + qb * C::BM;
          bulk_load(smem + C::OFF_VEC + slot * 1024, args.lse2 + voff, 512, &q_full[slot]);
          bulk_load(smem + C::OFF_VEC + slot * 1024 + 512, args.delta + voff, 512, &q_full[slot]);
          if (it == 0) {
            if (ci > 0 && !(ok = mbar_wait(mma_done, (ci - 1) & 1, abort_flag))) {
              kn = ci + 1, vn = ci, qn = p + 1, dn = p;
              break;
            }
            mbar_arrive_expect_tx(v_full, C::TILE);
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_3d(smem + vbuf + c * C::SUB, &tmV, v_full, c * 64, ky, kz);
          }
          if (p > 0 && !(ok = mbar_wait(do_empty, (p - 1) & 1, abort_flag))) {
            kn = vn = ci + 1, qn = p + 1, dn = p;
            break;
          }
          mbar_arrive_expect_tx(do_full, C::TILE);
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_3d(smem + C::OFF_DO + c * C::SUB, &tmDO, do_full, c * 64, qy, qz);
        }
        pc += wk.n_iter;
        if (!ok) {
          ++ci;
          break;
        }
      }
      if (kn < 0) kn = vn = ci, qn = dn = pc;  // every load of the items begun was issued
      // Do not leave with copies in flight (matters only after an abort, when
      // the consumers stopped waiting): the last load issued on each barrier
      // (each one was issued, so it lands and the bound is not reached).
      if (kn > 0) mbar_wait_drain(k_full, (kn - 1) & 1);
      if (vn > 0) mbar_wait_drain(v_full, (vn - 1) & 1);
      for (int p = max(0, qn - 2); p < qn; ++p) mbar_wait_drain(&q_full[p & 1], (p >> 1) & 1);
      if (dn > 0) mbar_wait_drain(do_full, (dn - 1) & 1);
    }
  } else if (warp == 1 || warp == 14) {
    // ---------------------------------------------------------------- MMA
    // Two issuing threads: warp 1 issues S^T, dV and dP^T (the chain the key
    // rows wait on), warp 14 issues dK and dQ once dS^T is ready, so neither
    // queue of products waits behind the other's issue. (The deterministic
    // order keeps warp 14 for its reductions: warp 1 then issues everything.)
    const bool do_a = warp == 1;
    const bool do_b = DET || warp == 14;
    if (!DET || warp == 1) {
      // The whole warp runs the issuing loop (warp-uniform waits), one elected
      // lane issues and commits.
      auto wwait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      constexpr uint32_t ID_SS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t ID_ACC = idesc_bf16_f32(128, D, false, true);    // dV, dK
      constexpr uint32_t ID_DQ = idesc_bf16_f32(128, D, true, true);      // dQ
      const uint32_t sb = smem_u32(smem);
      // Operand descriptors are built once, K-major (k*) and MN-major (m*); a
      // Q slot or a k-step only advances the start address (sdesc_advance).
      auto kd = [&](uint32_t off) { return sdesc_sw128(sb + off, 16, 1024); };
      auto md = [&](uint32_t off) { return sdesc_sw128(sb + off, C::SUB, 1024); };
      // K and V alternate between two buffers from item to item (see the TMA warp).
      const uint64_t kB0 = kd(C::OFF_K), kB1 = kd(C::OFF_V), kQ = kd(C::OFF_Q), kDO = kd(C::OFF_DO);
      const uint64_t mB0 = md(C::OFF_K), mB1 = md(C::OFF_V), mQ = md(C::OFF_Q), mDO = md(C::OFF_DO),
                     mDS = md(C::OFF_DS);
      auto kstep = [](int kk) { return static_cast<uint32_t>((kk >> 2) * C::SUB + (kk & 3) * 32); };  // 16 along K
      auto mstep = [](int kk) { return static_cast<uint32_t>(kk * 16 * 128); };                        // 16 K rows
      // X^T = A_rows(K-major, D) * B_rows(K-major, D)^T into a 128-column region
      auto issue_t = [&](uint32_t dst, uint64_t a, uint64_t b) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss_w(dst, sdesc_advance(a, kstep(kk)), sdesc_advance(b, kstep(kk)), ID_SS, kk > 0);
      };
      // One TMEM region per block pair p (X = R[p%2]) holds in turn S^T_p,
      // P^T_p, dP^T_p and dQ_p; the other region (Y) already takes S^T_(p+1)
      // while the key-row warpgroups compute dS^T_p.
      bool ok = true;
      int ci = 0, pc = 0;
      for (;; ++ci) {
        const int w = take_item_warp(ci);
        if (w < 0) break;
        const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, w);
        const bool swap = ci & 1;
        const uint64_t kK = swap ? kB1 : kB0, kV = swap ? kB0 : kB1, mK = swap ? mB1 : mB0;
        // Only the S^T issuer waits for K: dK and dQ follow ds_ready, which the
        // key rows arrive on after S^T (hence after this wait). The next item's
        // K may land before the other issuer has finished this one, so a wait
        // there could find the barrier two phases on.
        ok = !do_a || wwait(k_full, ci & 1);
        if (do_a && ok) {
          // S^T of the item's first pair: its region was released by the dQ
          // warpgroup (dq_empty of pair pc - 2), waited for after dP^T_(pc-1).
          ok = wwait(&q_full[pc & 1], (pc >> 1) & 1);
          tc_fence_after();
          issue_t((pc & 1) ? tR1 : tR0, kK, sdesc_advance(kQ, (pc & 1) * C::TILE));
          tc_commit_w(s_full);
        }
        for (int it = 0; it < wk.n_iter && ok; ++it) {
          const int p = pc + it;
          const int slot = p & 1;
          const uint32_t tx = (p & 1) ? tR1 : tR0;  // S/P^T, then dP^T, then dQ of pair p
          const uint32_t ty = (p & 1) ? tR0 : tR1;  // S^T of pair p+1
          const uint64_t mQs = sdesc_advance(mQ, slot * C::TILE);
          if (do_a) {
            // The first dV of an item restarts the accumulator: p_ready of its
            // first pair comes from the key rows after they have read the
            // previous item's dV and dK out of TMEM.
            if (it == 0) ok = wwait(v_full, ci & 1);
            ok = ok && wwait(do_full, p & 1) && wwait(p_ready, p & 1);
            tc_fence_after();
            // dV += P^T dO_p; P^T of query half h sits at columns [64h, 64h+32).
#pragma unroll
            for (int kk = 0; kk < C::BM / 16; ++kk)
              tc_mma_ts_w(tDV, tx + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(mDO, mstep(kk)), ID_ACC,
                          (it > 0 || kk > 0) ? 1u : 0u);
            // dP^T_p over the P^T it has just consumed (in-order tensor pipe).
            issue_t(tx, kV, kDO);
            tc_commit_w(dp_full);
            tc_commit_w(do_empty);
            // Region Y is free once the dQ warpgroup has read dQ_(p-1) out of
            // it. Waiting here, after every pair (the last of an item too), also
            // keeps dQ_p from completing before dQ_(p-1) is taken, which the
            // single issuer of the deterministic order relies on.
            if (p > 0) ok = ok && wwait(dq_empty, (p - 1) & 1);
            if (it + 1 < wk.n_iter) {
              const int ns = (p + 1) & 1;
              ok = ok && wwait(&q_full[ns], ((p + 1) >> 1) & 1);
              tc_fence_after();
              issue_t(ty, kK, sdesc_advance(kQ, ns * C::TILE));
              tc_commit_w(s_full);
            }
          }
          if (!do_b) continue;
          // dQ_p must not complete before the dQ warpgroup has taken dQ_(p-1)
          // (with one issuing thread the wait above already covers it). The
          // first dK of an item follows ds_ready, like dV after p_ready.
          if (!do_a && p > 0) ok = ok && wwait(dq_empty, (p - 1) & 1);
          ok = ok && wwait(ds_ready, p & 1);
          tc_fence_after();
          // dK += dS^T Q_p with dS^T read from X (laid out like P^T): the A
          // operand from TMEM saves shared-memory bandwidth, the kernel's limit ...
#pragma unroll
          for (int kk = 0; kk < C::BM / 16; ++kk)
            tc_mma_ts_w(tDK, tx + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(mQs, mstep(kk)), ID_ACC,
                        (it > 0 || kk > 0) ? 1u : 0u);
          tc_commit_w(&q_empty[slot]);
          // ... before dQ_p = dS K_j overwrites X (A = dS^T in SMEM read as MN-major)
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            tc_mma_ss_w(tx, sdesc_advance(mDS, mstep(kk)), sdesc_advance(mK, mstep(kk)), ID_DQ, kk > 0);
          tc_commit_w(dq_full);
          tc_commit_w(ds_free);  // the dS^T buffer may take dS^T_(p+1)
        }
        tc_commit_w(mma_done);
        pc += wk.n_iter;
        if (!ok) {
          ++ci;
          break;
        }
      }
      // Every product this thread issued has completed before the TMEM is
      // released, also after an abort (the other issuer does the same, and
      // the release follows a CTA barrier).
      uint64_t* fin_bar = &fin[warp == 1 ? 0 : 1];
      tc_commit_w(fin_bar);
      mbar_wait_drain(fin_bar, 0);
    } else if (DET && lane == 0) {
      // ----------------------- deterministic order only: dQ reduction issuer
      // The key blocks that see dQ tile qb are 0..jmax; they add their shares
      // in descending order, so block j goes after the jmax - j blocks above it.
      // Causal: block j+1 reaches every tile one step before block j (its first
      // tile is one higher) and started no later, so its share is normally in by
      // the time j gets there; waiting here for the completion of this block's
      // additions keeps that latency off the readout warps. Items are claimed
      // in ticket order and a block only waits for blocks with smaller tickets
      // (claimed earlier, by CTAs that are running), so the waits always end.
      const float4* stage = reinterpret_cast<const float4*>(smem + C::OFF_STAGE);
      int pc = 0;
      for (int ci = 0;; ++ci) {
        const int w = take_item(ci);
        if (w < 0) break;
        const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, w);
        bool ok = true;
        for (int it = 0; it < wk.n_iter && ok; ++it) {
          const int p = pc + it;
          const int qb = wk.i_lo + it;
          int jmax = (wk.sv.Lk + C::BN - 1) / C::BN - 1;
          if (CAUSAL) jmax = min(jmax, (qb * C::BM + C::BM - 1 + wk.sv.shift) / C::BN);
          uint32_t* turn = args.dq_turn + static_cast<size_t>(wk.bh) * nqb + qb;
          if (!counter_wait_eq(turn, static_cast<uint32_t>(jmax - wk.j), abort_flag)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          const size_t tile0 = (static_cast<size_t>(wk.bh) * nqb + qb) * C::HALVES;
          // The tile goes out in 32-column quarters (16 KB), alternately from
          // the two staging buffers; a buffer is handed back once the next
          // quarter's reduction is under way and its own has been read.
          constexpr int QPT = 2 * C::HALVES;  // quarters per tile
          for (int k = 0; k < QPT; ++k) {
            const int qn = p * QPT + k;  // quarters staged so far, over all items
            const int bsel = qn & 1;
            if (!mbar_wait(stage_full[bsel], (qn >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            bulk_reduce_add_f32(args.dq_acc + (tile0 + (k >> 1)) * (128 * 64) + (k & 1) * (8 * 128 * 4),
                                stage + bsel * (8 * 128), 16384);
            bulk_commit_group();
            if (k > 0) {
              bulk_wait_group_read<1>();  // the previous quarter's buffer has been read
              mbar_arrive(stage_free[bsel ^ 1]);
            }
          }
          if (!ok) break;
          bulk_wait_group<0>();  // this block's additions to tile qb are complete
          mbar_arrive(stage_free[(p * QPT + QPT - 1) & 1]);
          fence_proxy_async_global();
          red_release_gpu_add(turn, 1u);
        }
        pc += wk.n_iter;
        if (!ok) break;
      }
      bulk_wait_group<0>();
    }
  } else if (warp < 10) {
    // ------------------- key rows: P^T, dS^T for query half h, dK/dV epilogue
    const int h = (warp - 2) >> 2;  // query columns [64h, 64h+64)
    const int kk = (warp & 3) * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = sh.scale_log2;
    uint8_t* ds_row = smem + C::OFF_DS + h * C::SUB + kk * 128;
    bool ok = true;
    int pc = 0;
    for (int ci = 0; ok; ++ci) {
      const int w = take_item_warp(ci);
      if (w < 0) break;
      const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, w);
      const int key = wk.key0 + kk;
      const bool kvalid = key < wk.sv.Lk;
      for (int it = 0; it < wk.n_iter && ok; ++it) {
        const int p = pc + it;
        const int slot = p & 1;
        const uint32_t tr = ((p & 1) ? tR1 : tR0) + lo;  // S^T, then P^T, then dP^T of pair p
        const uint32_t tp = tr;
        const int qb = wk.i_lo + it;
        // Masked pairs: key key0+kk is hidden from query qb*128+qa iff qa < lim.
        // Fixed layout (no shift): only the diagonal pair qb == j has masked
        // pairs, with lim = kk.
        const int lim = VARLEN ? key - wk.sv.shift - qb * C::BM : kk;
        const bool diag = CAUSAL && (VARLEN ? lim > 0 : qb == wk.j);
        const float* lse2v = reinterpret_cast<const float*>(smem + C::OFF_VEC + slot * 1024) + h * 64;
        const float* deltav = lse2v + 128;
        ok = mbar_wait(s_full, p & 1, abort_flag) && mbar_wait(&q_full[slot], (p >> 1) & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);  // warp-collective TMEM accesses follow
        if (!ok) break;
        tc_fence_after();
        // P^T = 2^(S^T * sl2 + nlse2) for 64 queries, 32 at a time; P stays in
        // registers (bf16 pairs) for dS and goes to TMEM for the dV product.
        uint32_t pk[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t s[32];
          tmem_ld32(tr + h * 64 + c * 32, s);
          tmem_wait_ld();
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2v + c * 32 + q4 * 4);  // -LSE*log2(e)
            const uint64_t lp[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int q = q4 * 2 + e;
              const int qa = h * 64 + c * 32 + 2 * q;  // query column within the block
              float xa, xb;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * q]), __uint_as_float(s[2 * q + 1])), sl2x2, lp[e]), xa, xb);
              float pa = ex2(xa);
              float pb = ex2(xb);
              if (!kvalid) pa = pb = 0.f;
              if (diag) {
                if (qa < lim) pa = 0.f;
                if (qa + 1 < lim) pb = 0.f;
              }
              pk[c][q] = pack_bf16x2(pa, pb);
            }
          }
          tmem_st16(tr + h * 64 + c * 16, pk[c]);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_ready);
        // dS^T = P^T o (dP^T - delta) -> bf16 into the swizzled key-major
        // buffer, once dQ_(p-1) (issued by the other thread) has read the
        // previous dS^T out of it. That is checked first, while dP^T_p is
        // still running: dQ_(p-1) was issued long before, so the check costs
        // nothing on the path from dp_full to the dS^T math.
        ok = __all_sync(0xffffffffu, (p == 0 || mbar_wait(ds_free, (p - 1) & 1, abort_flag)) &&
                                         mbar_wait(dp_full, p & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dp[32];
          tmem_ld32(tp + h * 64 + c * 32, dp);
          tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 d4 = *reinterpret_cast<const float4*>(deltav + c * 32 + q4 * 4);
            const uint64_t dlt[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int q = q4 * 2 + e;
              const uint64_t pp = f2_pack(__uint_as_float(pk[c][q] << 16), __uint_as_float(pk[c][q] & 0xFFFF0000u));
              const uint64_t dd = f2_pack(__uint_as_float(dp[2 * q]), __uint_as_float(dp[2 * q + 1]));
              float da, db;
              f2_unpack(f2_mul(pp, f2_sub(dd, dlt[e])), da, db);
              w[q] = pack_bf16x2(da, db);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = (c * 4 + u) ^ (kk & 7);
            *reinterpret_cast<uint4*>(ds_row + unit * 16) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
          tmem_st16(tr + h * 64 + c * 16, w);  // over dP^T columns already read
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ds_ready);
      }
      pc += wk.n_iter;
      if (!ok) break;
      // ---------------------------------------------- dK, dV epilogue (half h of the columns)
      ok = __all_sync(0xffffffffu, mbar_wait(mma_done, ci & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      if constexpr (VARLEN) {
        // Packed layout (many short items: about 57 per CTA on a batch of 16
        // sequences of 512..8192 tokens): each thread writes its own half row
        // straight to global memory, without the two barriers of the staged
        // form below, which cost 3 % there while saving 2 % on long items.
        // Rows past this sequence belong to the next one.
        const bool store = key < wk.sv.Lk;
        const size_t roff = k_row<VARLEN>(args.pk, sh, wk.sv, wk.bh, key) * D;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t tacc = (which == 0 ? tDV : tDK) + lo;
          const float mul = which == 0 ? 1.f : sh.scale;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(which == 0 ? args.dv : args.dk) + roff);
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            const int c = h * (D / 64) + cc;  // 32-column chunk index
            uint32_t v[32];
            tmem_ld32(tacc + c * 32, v);
            tmem_wait_ld();
            if (store) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint4 x;
                x.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
                x.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
                x.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
                x.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
                dst[c * 4 + u] = x;
              }
            }
          }
        }
      } else {
        // Each of dV and dK goes out through the dS^T buffer (free: every product
        // of the item has completed), written there in the same swizzled key-major
        // layout by its key-row thread, then copied to global memory as whole row
        // segments by all 256 key-row threads (8 threads per 128-byte segment).
        // Fixed layout: keys past kv_len (< N) get their zero gradients written
        // (the accumulators hold zero there: every P^T and dS^T entry of such a
        // key is masked); packed layout: rows past this sequence belong to the
        // next one.
        const int ktid = threadIdx.x - 64;  // 0..255 over the key-row warps
        uint8_t* stage = smem + C::OFF_DS;
        auto srow = [&](int row, int g) {  // 16-byte unit g (8 columns) of key row `row`
          return stage + (g >> 3) * C::SUB + row * 128 + (((g & 7) ^ (row & 7)) << 4);
        };
  #pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t tacc = (which == 0 ? tDV : tDK) + lo;
          const float mul = which == 0 ? 1.f : sh.scale;
  #pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            const int c = h * (D / 64) + cc;  // 32-column chunk index
            uint32_t v[32];
            tmem_ld32(tacc + c * 32, v);
            tmem_wait_ld();
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 x;
              x.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
              x.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
              x.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
              x.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
              *reinterpret_cast<uint4*>(srow(kk, c * 4 + u)) = x;
            }
          }
          // A barrier of the 256 key-row threads, made of an mbarrier so that the
          // wait is bounded (a warp that gave up earlier never arrives).
          const uint32_t ep = (2 * ci + which) & 1;
          mbar_arrive(epi_full);
          ok = __all_sync(0xffffffffu, mbar_wait(epi_full, ep, abort_flag));
          if (!ok) break;
          uint16_t* out = static_cast<uint16_t*>(which == 0 ? args.dv : args.dk);
          constexpr int G8 = D / 8;  // 16-byte units per row
  #pragma unroll
          for (int e = ktid; e < C::BN * G8; e += 256) {
            const int row = e / G8, g = e % G8;
            const int key_r = wk.key0 + row;
            if (packed ? key_r < wk.sv.Lk : key_r < N)
              *reinterpret_cast<uint4*>(out + k_row<VARLEN>(args.pk, sh, wk.sv, wk.bh, key_r) * D + g * 8) =
                  *reinterpret_cast<const uint4*>(srow(row, g));
          }
          mbar_arrive(epi_empty);  // the buffer is read out before it is written again
          ok = __all_sync(0xffffffffu, mbar_wait(epi_empty, ep, abort_flag));
          if (!ok) break;
        }
        if (!ok) break;
      }
      // The next item's p_ready and ds_ready (each arrived after
      // tc_fence_before) order these TMEM reads before its first dV and dK.
    }
  } else if (warp == 15) {
    // ----------------- key blocks no query sees
    // Their dK and dV rows are zero: in the fixed layout the blocks past a
    // batch entry's key length, in a packed batch every key of a sequence
    // without queries. The main loop skips such items; this warp writes their
    // rows, in the background, for every item numbered blockIdx.x modulo the
    // grid (each row's 16-byte groups by consecutive lanes).
    {
      constexpr int G8 = D / 8;  // 16-byte groups per row
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int t = blockIdx.x; t < n_items; t += gridDim.x) {
        const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, t);
        if (wk.n_iter > 0) continue;
        const int rows = min(C::BN, (packed ? wk.sv.Lk : N) - wk.key0);
        for (int e = lane; e < rows * G8; e += 32) {
          const size_t off = k_row<VARLEN>(args.pk, sh, wk.sv, wk.bh, wk.key0 + e / G8) * G8 + e % G8;
          reinterpret_cast<uint4*>(args.dk)[off] = z;
          reinterpret_cast<uint4*>(args.dv)[off] = z;
        }
      }
    }
  } else if (warp < 14) {
    // ------------------------------------------ query rows: dQ_i readout
    const int qq = (warp & 3) * 32 + lane;
    const int tid = threadIdx.x - 320;  // 0..127 within this warpgroup
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float4* stage = reinterpret_cast<float4*>(smem + C::OFF_STAGE);
    int pc = 0;
    if constexpr (!DET) {
      // dQ_p goes out in 32-column quarters (16 KB each, contiguous in the
      // accumulator), staged alternately in the two halves of the staging
      // buffer: staging a quarter waits only for the reduction issued two
      // quarters earlier, and the TMEM region is released (dq_empty) after
      // two quarters instead of after a wait for a whole 32 KB reduction.
      int use = 0;  // quarters staged so far; buffer = use & 1
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        // One decision for the whole warpgroup (each warp takes the item on
        // its own): it shares named barriers below.
        const int w = take_item_warp(ci);
        if (!named_bar_and(2, 128, w >= 0)) break;
        const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, w);
        for (int it = 0; it < wk.n_iter; ++it) {
          const int p = pc + it;
          const uint32_t tr = ((p & 1) ? tR1 : tR0) + lo;
          if (!named_bar_and(2, 128, mbar_wait(dq_full, p & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const size_t tile0 = (static_cast<size_t>(wk.bh) * nqb + wk.i_lo + it) * C::HALVES;
          uint32_t v[64];
          auto stage_quarter = [&](size_t half_tile, int part, const uint32_t* src) {
            float4* buf = stage + (use & 1) * (8 * 128);
            if (use >= 2) {  // the reduction that last read this buffer must be done reading it
              if (tid == 0) bulk_wait_group_read<1>();
              named_bar_sync(1, 128);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
              buf[u * 128 + qq] = make_float4(__uint_as_float(src[4 * u]), __uint_as_float(src[4 * u + 1]),
                                              __uint_as_float(src[4 * u + 2]), __uint_as_float(src[4 * u + 3]));
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (tid == 0) {
              bulk_reduce_add_f32(args.dq_acc + half_tile * (128 * 64) + part * (8 * 128 * 4), buf, 16384);
              bulk_commit_group();
            }
            ++use;
          };
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh) {
            tmem_ld32(tr + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tr + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (hh == C::HALVES - 1) {
              tc_fence_before();
              mbar_arrive(dq_empty);  // TMEM region free for S^T_(p+2)
            }
            stage_quarter(tile0 + hh, 0, v);
            stage_quarter(tile0 + hh, 1, v + 32);
          }
        }
        pc += wk.n_iter;
      }
      // Before the CTA leaves, the reductions must have read the staging
      // buffer; their additions in L2 complete with the kernel.
      if (tid == 0) bulk_wait_group_read<0>();
    } else {
      // Deterministic order: the same readout, but the reductions are issued
      // by the issuer warp above, which also waits for their completion; this
      // warpgroup only fills the staging buffer when the issuer has read it.
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        const int w = take_item_warp(ci);
        if (!named_bar_and(2, 128, w >= 0)) break;  // one decision, as above
        const BwdWork wk = bwd_work<D, CAUSAL, VARLEN, DET>(args, w);
        for (int it = 0; it < wk.n_iter && ok; ++it) {
          const int p = pc + it;
          const uint32_t tr = ((p & 1) ? tR1 : tR0) + lo;
          if (!named_bar_and(2, 128, mbar_wait(dq_full, p & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t v[64];
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh) {
            tmem_ld32(tr + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tr + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (hh == C::HALVES - 1) {
              tc_fence_before();
              mbar_arrive(dq_empty);  // TMEM region free for dP^T_(p+1)
            }
            // Two 32-column quarters (16 KB each), alternately in the two
            // staging buffers, each once the reduction of the quarter that last
            // used its buffer has read it.
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const int qn = (p * C::HALVES + hh) * 2 + part;  // quarters staged so far
              const int bsel = qn & 1;
              if (qn >= 2)
                ok = named_bar_and(1, 128, tid != 0 || mbar_wait(stage_free[bsel], ((qn >> 1) - 1) & 1, abort_flag));
              if (!ok) break;
              float4* buf = stage + bsel * (8 * 128);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                buf[u * 128 + qq] = make_float4(__uint_as_float(v[32 * part + 4 * u]), __uint_as_float(v[32 * part + 4 * u + 1]),
                                                __uint_as_float(v[32 * part + 4 * u + 2]), __uint_as_float(v[32 * part + 4 * u + 3]));
              fence_proxy_async_smem();
              mbar_arrive(stage_full[bsel]);
            }
            if (!ok) break;
          }
        }
        pc += wk.n_iter;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Fixed scratch for the allocation-free backward entry point. Some callers
// cannot call cudaMalloc (or any allocating routine) at the point where they
// need the backward, e.g. code running inside a memory pool or allocator
// hook, or a host framework whose device memory is owned by another
// subsystem. For them the backward workspace lives in this static device
// array instead: every GPU that loads the library reserves it until the
// process exits. In host code the array's name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress, once per device (and
// again if the device's context was torn down and recreated, e.g. after
// cudaDeviceReset: the module is then loaded anew and the array may move).
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Unique id of the calling thread's current context (0 if the driver cannot
// tell), through the driver entry points the runtime exposes.
static unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

cudaError_t noalloc_scratch(void** ptr, size_t* bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  e = cudaSetDevice(dev);  // binds (and if needed creates) the device's primary context
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with `dev` current
    if (e != cudaSuccess) return e;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *ptr = addr[dev];
  *bytes = kNoAllocScratchBytes;
  return cudaSuccess;
}

cudaError_t set_bwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_bwd_status() { return take_status_here(); }

// A device attribute of the current device (0 if unknown), read once per device.
template <cudaDeviceAttr ATTR>
static long long device_attr() {
  constexpr int kMaxDevices = 64;
  static std::atomic<long long> cached[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  long long v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int x = 0;
    if (cudaDeviceGetAttribute(&x, ATTR, dev) != cudaSuccess) return 0;
    v = x;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}
static long long l2_cache_bytes() { return device_attr<cudaDevAttrL2CacheSize>(); }
static long long sm_count() { return device_attr<cudaDevAttrMultiProcessorCount>(); }

template <int D, bool CAUSAL, bool VARLEN, bool DET>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdArgs& args, cudaStream_t stream,
                                const LaunchMarks* marks) {
  using C = BwdCfg<D>;
  const int N = args.s.N;
  const int nkb = (args.s.Nk + C::BN - 1) / C::BN;  // key blocks: one CTA each per head
  const int Npad = (N + C::BM - 1) / C::BM * C::BM;
  const long long BH = static_cast<long long>(args.s.B) * args.s.H;
  // Heads per group: at most as many as keep their Q and dO tiles (bf16) and
  // dQ accumulator (fp32), D * 8 bytes per padded row, within the L2 (on a
  // GB300, 32 heads at N = 4096, d = 128; more overflow it and slow the
  // kernel); groups of equal size.
  BwdArgs a = args;
  {
    const long long per_head = static_cast<long long>(Npad) * D * 8;
    const long long l2 = l2_cache_bytes();
    const long long g = l2 > 0 ? l2 / per_head : 16;
    a.heads_per_group = balanced_heads_per_group(BH, g);
  }
  constexpr int TPR = D / 8;
  // The three kernels are launched with programmatic stream serialization:
  // each may start while the kernel before it on the stream finishes (its
  // set-up overlaps that kernel's last CTAs) and waits (griddepcontrol.wait)
  // before it reads that kernel's results. With per-kernel timing events the
  // launches stay plain, so each event pair brackets one kernel alone.
  const bool pdl = marks == nullptr;
  {
    const long long threads = BH * Npad * TPR;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    mark(marks, true, 0, stream);
    cudaError_t e = launch_maybe_pdl(fa_bwd_pre_kernel<D, VARLEN>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                                     0, stream, pdl, a, Npad);
    mark(marks, false, 0, stream);
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = fa_bwd_kernel<D, CAUSAL, VARLEN, DET>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // Persistent: one CTA per SM (the kernel's shared memory admits one),
    // taking work items from the ticket counter the pre-pass has zeroed.
    const long long items = BH * nkb;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const long long sms = sm_count();
    const long long blocks = std::max<long long>(1, std::min<long long>(items, sms > 0 ? sms : 1));
    mark(marks, true, 1, stream);
    e = launch_maybe_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(C::THREADS), C::SMEM_BYTES, stream, pdl, tq,
                         tk, tv, tdo, a);
    mark(marks, false, 1, stream);
    if (e != cudaSuccess) return e;
  }
  {
    const long long blocks = BH * (Npad / C::BM) * (D / 64);  // one per 32 KB accumulator tile
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    mark(marks, true, 2, stream);
    cudaError_t e = launch_maybe_pdl(fa_bwd_dq_kernel<D, VARLEN>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     stream, pdl, a, Npad);
    mark(marks, false, 2, stream);
    return e;
  }
}

template <int D, bool CAUSAL, bool VARLEN>
static cudaError_t launch_bwd_order(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream,
                                    const LaunchMarks* m) {
  return a.deterministic ? launch_bwd_t<D, CAUSAL, VARLEN, true>(tq, tk, tv, tdo, a, stream, m)
                         : launch_bwd_t<D, CAUSAL, VARLEN, false>(tq, tk, tv, tdo, a, stream, m);
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const BwdArgs& a, cudaStream_t stream, const LaunchMarks* m) {
  const bool c = a.s.causal != 0;
  if (a.pk.varlen) {
    if (a.s.D == 64)
      return c ? launch_bwd_order<64, true, true>(tq, tk, tv, tdo, a, stream, m)
               : launch_bwd_order<64, false, true>(tq, tk, tv, tdo, a, stream, m);
    return c ? launch_bwd_order<128, true, true>(tq, tk, tv, tdo, a, stream, m)
             : launch_bwd_order<128, false, true>(tq, tk, tv, tdo, a, stream, m);
  }
  if (a.s.D == 64)
    return c ? launch_bwd_order<64, true, false>(tq, tk, tv, tdo, a, stream, m)
             : launch_bwd_order<64, false, false>(tq, tk, tv, tdo, a, stream, m);
  return c ? launch_bwd_order<128, true, false>(tq, tk, tv, tdo, a, stream, m)
           : launch_bwd_order<128, false, false>(tq, tk, tv, tdo, a, stream, m);
}

}  // namespace fa
