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
//   bwd_main     one CTA per (b, h, 128-key block j); loops over the 128-query
//                blocks i that see block j (causal: i >= j), all in TMEM/SMEM:
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
// Warp roles of bwd_main (15 warps): warp 0 TMA producer, warp 1 tcgen05
// issuer of S^T, dV and dP^T, warp 14 issuer of dK and dQ, warps 2-5 and 6-9
// one key row per thread for query columns 0-63 and 64-127 (P^T, dS^T, then
// half of the dK/dV epilogue each), warps 10-13 one query row per thread (dQ_i
// readout and reduction). Any four consecutive warps cover the four TMEM lane
// quarters (warp w reads lanes 32*(w%4)..+31). In the deterministic order
// warp 1 issues every product and warp 14 issues the dQ reductions in a fixed
// order across CTAs (see the dQ reduction issuer).
//
// dQ accumulator layout (private to the library): per (b*h, 128-query block,
// 64-column half) a 32 KB tile stored as [16 float4 column groups][128 rows],
// so the staging writes in shared memory are bank-conflict free and each half
// is one contiguous bulk reduction.
#include <mutex>

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
  static constexpr int OFF_STAGE = OFF_DS + 2 * SUB;   // dQ staging: 128 rows x 64 fp32 = 32 KB
  static constexpr int OFF_VEC = OFF_STAGE + 32768;    // 2 slots x (nlse2[128], delta[128]) fp32
  static constexpr int OFF_BAR = OFF_VEC + 2 * 1024;
  static constexpr int NUM_BARS = 16;
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16;
  static constexpr int THREADS = 480;
  static constexpr uint32_t TMEM_COLS = 512;
};

// Index (in floats) of element (row r, column c) of query block qb of head bh
// in the dQ accumulator.
__device__ __forceinline__ size_t dq_acc_index(int D, size_t bh, int nqb, int qb, int r, int c) {
  const size_t tile = (bh * nqb + qb) * static_cast<size_t>(D / 64) + (c >> 6);
  return ((tile * 16 + ((c & 63) >> 2)) * 128 + r) * 4 + (c & 3);
}

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
  // Counters of the deterministic order: one per 128-row block, and the ticket.
  if (tid < rows / 128) a.dq_turn[tid] = 0u;
  if (tid == 0) *a.ticket = 0u;
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
  // The accumulator has exactly D floats per padded row: zero them linearly.
  float4* z = reinterpret_cast<float4*>(a.dq_acc + row * D + g * 8);
  z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// dQ = scale * dq_acc -> bf16. Thread = (row, 8 columns); consecutive threads
// take consecutive rows so the accumulator reads are contiguous.
// ---------------------------------------------------------------------------
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdArgs a, int Npad) {
  constexpr int GROUPS = D / 8;
  const int N = a.s.N;
  const int nqb = Npad / 128;
  const size_t per_head = static_cast<size_t>(Npad) * GROUPS;
  const size_t total = static_cast<size_t>(a.s.B) * a.s.H * per_head;
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= total) return;
  const size_t bh = tid / per_head;
  size_t rem = tid % per_head;
  const int qb = static_cast<int>(rem / (128 * GROUPS));
  rem %= 128 * GROUPS;
  const int g = static_cast<int>(rem / 128);
  const int r = static_cast<int>(rem % 128);
  const int n = qb * 128 + r;
  const SeqView sv = seq_view<VARLEN>(a.pk, a.kv_lens, static_cast<int>(bh / a.s.H), N);
  if (n >= sv.Lq) return;
  const float4 x = *reinterpret_cast<const float4*>(a.dq_acc + dq_acc_index(D, bh, nqb, qb, r, g * 8));
  const float4 y = *reinterpret_cast<const float4*>(a.dq_acc + dq_acc_index(D, bh, nqb, qb, r, g * 8 + 4));
  const float s = a.s.scale;
  uint4 w;
  w.x = pack_bf16x2(x.x * s, x.y * s);
  w.y = pack_bf16x2(x.z * s, x.w * s);
  w.z = pack_bf16x2(y.x * s, y.y * s);
  w.w = pack_bf16x2(y.z * s, y.w * s);
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dq) + q_row<VARLEN>(a.pk, a.s, sv, static_cast<int>(bh), n) * D + g * 8) = w;
}

// ---------------------------------------------------------------------------
// Main kernel
// ---------------------------------------------------------------------------
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
  uint64_t* kv_full = bars + 0;
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
  uint64_t* mma_done = bars + 13;
  uint64_t* stage_full = bars + 14;  // deterministic order: 128 arrivals
  uint64_t* stage_free = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Deterministic order: work items are handed out by a global ticket in grid
  // order, so every item with a smaller ticket belongs to a CTA that has
  // already started; such a CTA finishes without waiting for a larger ticket
  // (it only ever waits for key blocks above its own, which come first).
  int item = blockIdx.x;
  if constexpr (DET) {
    volatile int* ticket_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);
    if (threadIdx.x == 0) *ticket_slot = static_cast<int>(atomicAdd(args.ticket, 1u));
    __syncthreads();
    item = *ticket_slot;
  }
  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int nkb = (sh.Nk + C::BN - 1) / C::BN;  // key blocks (grid)
  const int nqb = (N + C::BM - 1) / C::BM;       // query blocks of the padded workspace
  const int Npad = nqb * C::BM;
  // Groups of up to 16 heads run together, so their Q, dO and dQ accumulators
  // stay in L2; inside a group the key blocks go heaviest first (causal:
  // block j sees nkb - j query blocks) across the group's heads.
  const int BH = sh.B * sh.H;
  const int G = BH < 16 ? BH : 16;
  const int group = item / (G * nkb);
  const int gsize = min(G, BH - group * G);
  const int r_in = item - group * G * nkb;
  // Default order: heaviest key block first (causal: block j sees nkb - j query
  // blocks). Deterministic order: lightest first, see the dQ warpgroup.
  const int j = DET ? nkb - 1 - r_in / gsize : r_in / gsize;
  const int bh = group * G + r_in % gsize;
  const int b = bh / sh.H;
  const SeqView sv = seq_view<VARLEN>(args.pk, args.kv_lens, b, N);
  const int klim = sv.Lk;
  constexpr bool packed = VARLEN;
  const int head = bh % sh.H;
  const int key0 = j * C::BN;
  // Query r sees key c iff c <= r + shift (causal): the first query block that
  // sees key block j starts at row key0 - shift.
  // (Fixed layout: shift 0, every sequence nkb query blocks long.)
  const int i_lo = CAUSAL ? (VARLEN ? max(0, key0 - sv.shift) / C::BM : j) : 0;
  const int nq = VARLEN ? (sv.Lq + C::BM - 1) / C::BM : nkb;  // query blocks of this sequence
  const int n_iter = (key0 >= klim) ? 0 : (VARLEN ? max(0, nq - i_lo) : nkb - i_lo);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NUM_BARS; ++i) mbar_init(&bars[i], 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_empty, 128);
    mbar_init(mma_done, DET ? 1 : 2);  // one commit per issuing thread
    if (DET) mbar_init(stage_full, 128);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && n_iter > 0 && !g_test_drop_loads) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c) {
        const int y = packed ? head : key0, z = packed ? sv.k_start + key0 : bh;
        tma_load_3d(smem + C::OFF_K + c * C::SUB, &tmK, kv_full, c * 64, y, z);
        tma_load_3d(smem + C::OFF_V + c * C::SUB, &tmV, kv_full, c * 64, y, z);
      }
      for (int it = 0; it < n_iter; ++it) {
        const int slot = it & 1, use = it >> 1;
        const int qb = i_lo + it;
        const int qy = packed ? head : qb * C::BM, qz = packed ? sv.q_start + qb * C::BM : bh;
        if (use > 0 && !mbar_wait(&q_empty[slot], (use - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&q_full[slot], C::TILE + 1024);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(smem + C::OFF_Q + slot * C::TILE + c * C::SUB, &tmQ, &q_full[slot], c * 64, qy, qz);
        const size_t voff = static_cast<size_t>(bh) * Npad + qb * C::BM;
        bulk_load(smem + C::OFF_VEC + slot * 1024, args.lse2 + voff, 512, &q_full[slot]);
        bulk_load(smem + C::OFF_VEC + slot * 1024 + 512, args.delta + voff, 512, &q_full[slot]);
        if (it > 0 && !mbar_wait(do_empty, (it - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(do_full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(smem + C::OFF_DO + c * C::SUB, &tmDO, do_full, c * 64, qy, qz);
      }
      // Do not leave with copies in flight (matters only after an abort).
      mbar_wait(kv_full, 0, abort_flag);
      for (int it = max(0, n_iter - 2); it < n_iter; ++it) mbar_wait(&q_full[it & 1], (it >> 1) & 1, abort_flag);
      mbar_wait(do_full, (n_iter - 1) & 1, abort_flag);
    }
  } else if (warp == 1 || (!DET && warp == 14)) {
    // ---------------------------------------------------------------- MMA
    // Two issuing threads: warp 1 issues S^T, dV and dP^T (the chain the key
    // rows wait on), warp 14 issues dK and dQ once dS^T is ready, so neither
    // queue of products waits behind the other's issue. (The deterministic
    // order keeps warp 14 for its reductions: warp 1 then issues everything.)
    const bool do_a = warp == 1;
    const bool do_b = DET || warp == 14;
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t ID_SS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t ID_ACC = idesc_bf16_f32(128, D, false, true);    // dV, dK
      constexpr uint32_t ID_DQ = idesc_bf16_f32(128, D, true, true);      // dQ
      const uint32_t sb = smem_u32(smem);
      // Operand descriptors are built once, K-major (k*) and MN-major (m*); a
      // Q slot or a k-step only advances the start address (sdesc_advance).
      auto kd = [&](uint32_t off) { return sdesc_sw128(sb + off, 16, 1024); };
      auto md = [&](uint32_t off) { return sdesc_sw128(sb + off, C::SUB, 1024); };
      const uint64_t kK = kd(C::OFF_K), kV = kd(C::OFF_V), kQ = kd(C::OFF_Q), kDO = kd(C::OFF_DO);
      const uint64_t mK = md(C::OFF_K), mQ = md(C::OFF_Q), mDO = md(C::OFF_DO), mDS = md(C::OFF_DS);
      auto kstep = [](int kk) { return static_cast<uint32_t>((kk >> 2) * C::SUB + (kk & 3) * 32); };  // 16 along K
      auto mstep = [](int kk) { return static_cast<uint32_t>(kk * 16 * 128); };                        // 16 K rows
      // X^T = A_rows(K-major, D) * B_rows(K-major, D)^T into a 128-column region
      auto issue_t = [&](uint32_t dst, uint64_t a, uint64_t b) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(dst, sdesc_advance(a, kstep(kk)), sdesc_advance(b, kstep(kk)), ID_SS, kk > 0);
      };
      // One TMEM region per block pair i (X = R[i%2]) holds in turn S^T_i,
      // P^T_i, dP^T_i and dQ_i; the other region (Y) already takes S^T_(i+1)
      // while the key-row warpgroups compute dS^T_i.
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      if (do_a) {
        ok = ok && mbar_wait(&q_full[0], 0, abort_flag);
        tc_fence_after();
        issue_t(tR0, kK, kQ);  // S^T_0
        tc_commit(s_full);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const int slot = it & 1;
        const uint32_t tx = (it & 1) ? tR1 : tR0;  // S/P^T, then dP^T, then dQ of pair i
        const uint32_t ty = (it & 1) ? tR0 : tR1;  // S^T of pair i+1
        const uint64_t mQs = sdesc_advance(mQ, slot * C::TILE);
        if (do_a) {
          ok = mbar_wait(do_full, it & 1, abort_flag) && mbar_wait(p_ready, it & 1, abort_flag);
          tc_fence_after();
          // dV += P^T dO_i; P^T of query half h sits at columns [64h, 64h+32).
#pragma unroll
          for (int kk = 0; kk < C::BM / 16; ++kk)
            tc_mma_ts(tDV, tx + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(mDO, mstep(kk)), ID_ACC,
                      (it > 0 || kk > 0) ? 1u : 0u);
          // dP^T_i over the P^T it has just consumed (in-order tensor pipe).
          issue_t(tx, kV, kDO);
          tc_commit(dp_full);
          tc_commit(do_empty);
          const bool more = it + 1 < n_iter;
          if (more) {  // S^T_(i+1) once dQ_(i-1) has been read out of region Y
            const int ns = (it + 1) & 1;
            if (it > 0) ok = ok && mbar_wait(dq_empty, (it - 1) & 1, abort_flag);
            ok = ok && mbar_wait(&q_full[ns], ((it + 1) >> 1) & 1, abort_flag);
            tc_fence_after();
            issue_t(ty, kK, sdesc_advance(kQ, ns * C::TILE));
            tc_commit(s_full);
          } else if (it > 0 && do_b) {
            // Last pair: dQ_i must not complete before the dQ warpgroup has taken
            // dQ_(i-1), or dq_full would advance two phases past its waiter.
            ok = ok && mbar_wait(dq_empty, (it - 1) & 1, abort_flag);
          }
        }
        if (!do_b) continue;
        // dQ_i must not complete before the dQ warpgroup has taken dQ_(i-1)
        // (with one issuing thread the wait above already covers it).
        if (!do_a && it > 0) ok = ok && mbar_wait(dq_empty, (it - 1) & 1, abort_flag);
        ok = ok && mbar_wait(ds_ready, it & 1, abort_flag);
        tc_fence_after();
        // dK += dS^T Q_i with dS^T read from X (laid out like P^T): the A
        // operand from TMEM saves shared-memory bandwidth, the kernel's limit ...
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          tc_mma_ts(tDK, tx + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(mQs, mstep(kk)), ID_ACC,
                    (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&q_empty[slot]);
        // ... before dQ_i = dS K_j overwrites X (A = dS^T in SMEM read as MN-major)
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_ss(tx, sdesc_advance(mDS, mstep(kk)), sdesc_advance(mK, mstep(kk)), ID_DQ, kk > 0);
        tc_commit(dq_full);
      }
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag);
    }
  } else if (warp < 10) {
    // ------------------- key rows: P^T, dS^T for query half h, dK/dV epilogue
    const int h = (warp - 2) >> 2;  // query columns [64h, 64h+64)
    const int kk = (warp & 3) * 32 + lane;
    const int key = key0 + kk;
    const bool kvalid = key < klim;
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = sh.scale_log2;
    uint8_t* ds_row = smem + C::OFF_DS + h * C::SUB + kk * 128;
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      const int slot = it & 1;
      const uint32_t tr = ((it & 1) ? tR1 : tR0) + lo;  // S^T, then P^T, then dP^T of pair i
      const uint32_t tp = tr;
      const int qb = i_lo + it;
      // Masked pairs: key key0+kk is hidden from query qb*128+qa iff qa < lim.
      // Fixed layout (no shift): only the diagonal pair qb == j has masked
      // pairs, with lim = kk.
      const int lim = VARLEN ? key0 + kk - sv.shift - qb * C::BM : kk;
      const bool diag = CAUSAL && (VARLEN ? lim > 0 : qb == j);
      const float* lse2v = reinterpret_cast<const float*>(smem + C::OFF_VEC + slot * 1024) + h * 64;
      const float* deltav = lse2v + 128;
      ok = mbar_wait(s_full, it & 1, abort_flag) && mbar_wait(&q_full[slot], (it >> 1) & 1, abort_flag);
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
      // dS^T = P^T o (dP^T - delta) -> bf16 into the swizzled key-major buffer.
      ok = __all_sync(0xffffffffu, mbar_wait(dp_full, it & 1, abort_flag));
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
    // ------------------------------------------------ dK, dV epilogue (half h of the columns)
    if (n_iter > 0 && ok) {
      ok = mbar_wait(mma_done, 0, abort_flag);
      tc_fence_after();
    }
    // Fixed layout: keys past kv_len (< N) get their zero gradients written;
    // packed layout: rows past this sequence belong to the next one.
    const bool store = packed ? key < klim : key < N;
    const size_t roff = k_row<VARLEN>(args.pk, sh, sv, bh, key) * D;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t tacc = (which == 0 ? tDV : tDK) + lo;
      const float mul = which == 0 ? 1.f : sh.scale;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(which == 0 ? args.dv : args.dk) + roff);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = h * (D / 64) + cc;  // 32-column chunk index
        uint32_t v[32];
        if (n_iter > 0) {
          tmem_ld32(tacc + c * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
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
  } else if (warp < 14) {
    // ------------------------------------------ query rows: dQ_i readout
    const int qq = (warp & 3) * 32 + lane;
    const int tid = threadIdx.x - 320;  // 0..127 within this warpgroup
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float4* stage = reinterpret_cast<float4*>(smem + C::OFF_STAGE);
    if constexpr (!DET) {
      // dQ_i goes out in 32-column quarters (16 KB each, contiguous in the
      // accumulator), staged alternately in the two halves of the staging
      // buffer: staging a quarter waits only for the reduction issued two
      // quarters earlier, and the TMEM region is released (dq_empty) after
      // two quarters instead of after a wait for a whole 32 KB reduction.
      int use = 0;  // quarters staged so far; buffer = use & 1
      for (int it = 0; it < n_iter; ++it) {
        const uint32_t tr = ((it & 1) ? tR1 : tR0) + lo;
        // One decision for the whole warpgroup: it shares named barriers below.
        if (!named_bar_and(2, 128, mbar_wait(dq_full, it & 1, abort_flag))) break;
        tc_fence_after();
        const size_t tile0 = (static_cast<size_t>(bh) * nqb + i_lo + it) * C::HALVES;
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
            mbar_arrive(dq_empty);  // TMEM region free for S^T_(it+2)
          }
          stage_quarter(tile0 + hh, 0, v);
          stage_quarter(tile0 + hh, 1, v + 32);
        }
      }
      if (tid == 0) bulk_wait_group<0>();
    } else {
      // Deterministic order: the same readout, but the reductions are issued
      // by the issuer warp below, which also waits for their completion; this
      // warpgroup only fills the staging buffer when the issuer has read it.
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        const uint32_t tr = ((it & 1) ? tR1 : tR0) + lo;
        if (!named_bar_and(2, 128, mbar_wait(dq_full, it & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t v[64];
#pragma unroll
        for (int hh = 0; hh < C::HALVES; ++hh) {
          tmem_ld32(tr + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tr + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          if (hh == C::HALVES - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty);  // TMEM region free for dP^T_(it+1)
          }
          const int use = it * C::HALVES + hh;  // uses of the staging buffer so far
          if (use > 0) ok = named_bar_and(1, 128, tid != 0 || mbar_wait(stage_free, (use - 1) & 1, abort_flag));
          if (!ok) break;
#pragma unroll
          for (int u = 0; u < 16; ++u)
            stage[u * 128 + qq] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                              __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
          fence_proxy_async_smem();
          mbar_arrive(stage_full);
        }
      }
    }
  } else if (DET && lane == 0) {
    // ----------------------- deterministic order only: dQ reduction issuer
    // The key blocks that see dQ tile qb are 0..jmax; they add their shares
    // in descending order, so block j goes after the jmax - j blocks above it.
    // Causal: block j+1 reaches every tile one step before block j (its first
    // tile is one higher) and started no later, so its share is normally in by
    // the time j gets there; waiting here for the completion of this block's
    // additions keeps that latency off the readout warps.
    const float4* stage = reinterpret_cast<const float4*>(smem + C::OFF_STAGE);
    for (int it = 0; it < n_iter; ++it) {
      const int qb = i_lo + it;
      int jmax = (klim + C::BN - 1) / C::BN - 1;
      if (CAUSAL) jmax = min(jmax, (qb * C::BM + C::BM - 1 + sv.shift) / C::BN);
      uint32_t* turn = args.dq_turn + static_cast<size_t>(bh) * nqb + qb;
      if (!counter_wait_eq(turn, static_cast<uint32_t>(jmax - j), abort_flag)) break;
      fence_proxy_async_global();
      const size_t tile0 = (static_cast<size_t>(bh) * nqb + qb) * C::HALVES;
      bool ok = true;
      for (int hh = 0; hh < C::HALVES; ++hh) {
        const int use = it * C::HALVES + hh;
        if (!mbar_wait(stage_full, use & 1, abort_flag)) {
          ok = false;
          break;
        }
        bulk_reduce_add_f32(args.dq_acc + (tile0 + hh) * (128 * 64), stage, 32768);
        bulk_commit_group();
        bulk_wait_group_read<0>();
        mbar_arrive(stage_free);
      }
      if (!ok) break;
      bulk_wait_group<0>();  // this block's additions to tile qb are complete
      fence_proxy_async_global();
      red_release_gpu_add(turn, 1u);
    }
    bulk_wait_group<0>();
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
// its device address comes from cudaGetSymbolAddress, once per device.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t noalloc_scratch(void** ptr, size_t* bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with `dev` current
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  *bytes = kNoAllocScratchBytes;
  return cudaSuccess;
}

cudaError_t set_bwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_bwd_status() { return take_status_here(); }

template <int D, bool CAUSAL, bool VARLEN, bool DET>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream,
                                const LaunchMarks* marks) {
  using C = BwdCfg<D>;
  const int N = a.s.N;
  const int nkb = (a.s.Nk + C::BN - 1) / C::BN;  // key blocks: one CTA each per head
  const int Npad = (N + C::BM - 1) / C::BM * C::BM;
  const long long BH = static_cast<long long>(a.s.B) * a.s.H;
  constexpr int TPR = D / 8;
  {
    const long long threads = BH * Npad * TPR;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    mark(marks, true, 0, stream);
    fa_bwd_pre_kernel<D, VARLEN><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a, Npad);
    mark(marks, false, 0, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = fa_bwd_kernel<D, CAUSAL, VARLEN, DET>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long blocks = BH * nkb;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    mark(marks, true, 1, stream);
    kern<<<static_cast<unsigned>(blocks), C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, a);
    mark(marks, false, 1, stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    const long long threads = BH * Npad * TPR;
    const long long blocks = (threads + 255) / 256;
    mark(marks, true, 2, stream);
    fa_bwd_dq_kernel<D, VARLEN><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a, Npad);
    mark(marks, false, 2, stream);
    return cudaGetLastError();
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
