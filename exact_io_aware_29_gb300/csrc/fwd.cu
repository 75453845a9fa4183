// Forward pass of exact attention on sm_103a.
//
// Computes, per (batch, head), O = softmax(scale * Q K^T + M) V and the row
// log-sum-exp, by tiling Q into 128-row blocks and scanning K/V in 128-row
// blocks with the online-softmax recurrence (running max m, denominator l,
// unnormalised accumulator, rescale factor alpha = 2^(m_old - m_new)), so the
// logits S and probabilities P never leave the SM.
//   Math: "FlashAttention算法详解：从IO瓶颈到Triton实现", §Online Softmax and
//   §FlashAttention Forward流程 (the loop), §Causal Mask怎么处理 (three block
//   classes: full / skipped / masked), §Backward为什么更复杂 (LSE = m + log l);
//   youngju.dev flash_attention.zh §8.1-8.3 (deferred normalisation, Q-block
//   parallelism, no inter-warp reduction).
//
// GB300 mapping (one CTA = two 128-row Q tiles of one (b, h)):
//   warp 0      TMA producer: Q tiles once, then K_j / V_j into a ring of
//               shared-memory slots (128B swizzle), mbarrier full/empty pairs.
//   warp 1      tcgen05 issuer (one thread): S_t = Q_t K_j^T into TMEM (bf16
//               inputs), then O_t += P_t V_j with P_t read from TMEM (aliasing
//               S_t); this second product runs in f16 (P and V both f16).
//   warps 2-3   convert each V_j tile in shared memory from bf16 to f16 in
//               place (exact for bf16 values in f16's normal range), so P can
//               be quantised to f16 (unit roundoff 2^-11) instead of bf16
//               (2^-8): the P quantisation is the largest error term of O.
//               They also track the largest magnitude among the CTA's V values.
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: one thread per
//               query row (TMEM lane), exp2-domain online softmax, P written
//               back to TMEM as f16, O rescaled in TMEM only when the running
//               max grows by more than 2^8 (exact: m, l and O share the same
//               reference max), then the epilogue O = acc / l and LSE.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
//
// Range of V. f16 holds bf16 values exactly only for magnitudes in
// [2^-14, 65536) (bf16 exponent fields 113..142; smaller values land on f16's
// subnormal grid, larger ones overflow). A CTA whose V values (over the keys
// below its key limit in every block it loads; the rest are zeroed) reach
// 65536, or all stay below 2^-14, repeats its whole
// scan in a second pass: there V is scaled in shared memory by 2^k (exact, the
// largest magnitude then lies in [2, 4)), P is quantised to bf16 (same
// exponent range as fp32) and P V runs with bf16 operands; the epilogue
// multiplies O by 2^-k. The first pass then only serves to find the range,
// and the common case pays nothing but the exponent tracking. P carries a
// factor 2^7 in both passes (folded into the exponent; l carries it too, so
// O = acc / l is unchanged and the LSE subtracts 7): with the lazy rescale P
// stays below 2^15, inside f16's range, and probabilities down to 2^-38 of
// the running maximum keep f16 normals instead of flushing to zero.
#include "common.cuh"
#include "ptx.cuh"

namespace fa {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                       // query rows per tile
  static constexpr int BN = 128;                       // keys per block
  static constexpr int QT = 2;                         // Q tiles per CTA
  static constexpr int CHUNKS = D / 64;                // 64-column (128 B) swizzle chunks
  static constexpr int STAGES = (D == 128) ? 4 : 8;    // K/V ring slots
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int SUB_BYTES = 128 * 128;          // one [128 rows x 64 cols] bf16 chunk
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = QT * Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * KV_BYTES;
  static constexpr int NUM_BARS = 2 + 3 * STAGES + 2 + 2 + 2 + 1 + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 384;
  static constexpr int CONV_WARP0 = 2;     // warps 2-3 convert V
  static constexpr int CONV_THREADS = 64;
  static constexpr uint32_t TMEM_COLS = 512;
};

// Second-pass decision from the largest bf16 magnitude (the 15 bits below the
// sign) among the V values a CTA loaded: returns the power-of-two shift k of V
// for the bf16 pass, or kNoSecondPass when the f16 pass was exact enough. An
// all-zero V and non-finite values (which make O non-finite in either pass)
// need no second pass. With e the largest exponent field, k = 128 - e puts the
// largest magnitude in [2, 4); k is capped at 126 (V made only of bf16
// subnormals) so that 2^k and 2^-k stay normal fp32 numbers.
constexpr int kNoSecondPass = 1 << 20;
__device__ __forceinline__ int v_second_pass_shift(uint32_t vmag, int n_max) {
  const int e = static_cast<int>(vmag >> 7);
  if (n_max == 0 || vmag == 0 || e == 255) return kNoSecondPass;
  if (e >= 113 && e <= 142) return kNoSecondPass;
  return min(128 - e, 126);
}

// 2^e as an fp32 constant, for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// p = 2^(s * sl2 - msub) for the 128 logits of one row (in registers),
// summed into rs0 / rs1 and written to TMEM over S as 64 packed f16 pairs.
__device__ __forceinline__ void softmax_exp_store_f16(const uint32_t (&s)[128], float sl2, float msub, float& rs0,
                                                      float& rs1, uint32_t tS) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float p0 = ex2(fmaf(__uint_as_float(s[h * 64 + 2 * i]), sl2, -msub));
      const float p1 = ex2(fmaf(__uint_as_float(s[h * 64 + 2 * i + 1]), sl2, -msub));
      rs0 += p0;
      rs1 += p1;
      pk[i] = pack_f16x2(p0, p1);
    }
    tmem_st32(tS + h * 32, pk);
  }
}

// The same for the (rare) bf16 second pass, as a compact loop: it re-reads
// the logits from TMEM 8 columns at a time (masked logits are re-masked from
// the key limit) and writes 4 packed bf16 pairs over the columns already
// read, so the first pass keeps the only fully unrolled copy.
__device__ __forceinline__ void softmax_exp_store_bf16(uint32_t tS, float sl2, float msub, int kb, int cmax,
                                                       float& r0, float& r1) {
#pragma unroll 1
  for (int c = 0; c < 16; ++c) {
    uint32_t x[8];
    tmem_ld8(tS + c * 8, x);
    tmem_wait_ld();
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k0 = kb + c * 8 + 2 * i;
      const float p0 = k0 < cmax ? ex2(fmaf(__uint_as_float(x[2 * i]), sl2, -msub)) : 0.f;
      const float p1 = k0 + 1 < cmax ? ex2(fmaf(__uint_as_float(x[2 * i + 1]), sl2, -msub)) : 0.f;
      r0 += p0;
      r1 += p1;
      pk[i] = pack_bf16x2(p0, p1);
    }
    tmem_st4(tS + c * 4, pk);
  }
}

// Converter loops over one V tile of 128 keys x D (``units`` 16-byte units,
// 64-column chunks of 128 rows of 128 bytes: each row holds one key, the 128B
// swizzle permutes 16-byte units within a row only). Thread ``ct`` of the CT
// converter threads handles units ct, ct + CT, ... With MASK, keys at or past
// ``rows_valid`` read as zero: they are masked for every query (P = 0), but
// the tile holds whatever the tensor has there (key padding, or the next
// sequence of a packed batch), and zeroed they can neither widen the range the
// CTA tracks nor turn 0 * V into NaN after an f16 overflow.
template <bool MASK>
__device__ __forceinline__ uint4 load_v_unit(const uint4* tile, int u, int rows_valid) {
  uint4 x = tile[u];
  if (MASK && ((u & 1023) >> 3) >= rows_valid) x = make_uint4(0u, 0u, 0u, 0u);
  return x;
}

// One packed bf16 pair -> packed f16 pair, folding both magnitudes into the
// running maximum ``vmax`` (one 3-input max on the unpacked values).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_track(uint32_t w, float& vmax) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  vmax = max3f(vmax, fabsf(lo), fabsf(hi));
  return pack_f16x2(lo, hi);
}

// First pass: bf16 -> f16 in place, tracking the largest magnitude (max
// ignores NaN; an infinity makes the maximum infinite).
template <bool MASK, int UNITS, int CT>
__device__ __forceinline__ void convert_v_f16(uint4* tile, int rows_valid, int ct, float& vmax) {
#pragma unroll 4
  for (int u = ct; u < UNITS; u += CT) {
    uint4 x = load_v_unit<MASK>(tile, u, rows_valid);
    x.x = bf16x2_to_f16x2_track(x.x, vmax);
    x.y = bf16x2_to_f16x2_track(x.y, vmax);
    x.z = bf16x2_to_f16x2_track(x.z, vmax);
    x.w = bf16x2_to_f16x2_track(x.w, vmax);
    tile[u] = x;
  }
}

// Second pass: bf16 * 2^k in place (f = 2^k), still bf16.
template <bool MASK, int UNITS, int CT>
__device__ __forceinline__ void scale_v_bf16(uint4* tile, int rows_valid, int ct, float f) {
  for (int u = ct; u < UNITS; u += CT) {
    uint4 x = load_v_unit<MASK>(tile, u, rows_valid);
    x.x = pack_bf16x2(__uint_as_float(x.x << 16) * f, __uint_as_float(x.x & 0xFFFF0000u) * f);
    x.y = pack_bf16x2(__uint_as_float(x.y << 16) * f, __uint_as_float(x.y & 0xFFFF0000u) * f);
    x.z = pack_bf16x2(__uint_as_float(x.z << 16) * f, __uint_as_float(x.z & 0xFFFF0000u) * f);
    x.w = pack_bf16x2(__uint_as_float(x.w << 16) * f, __uint_as_float(x.w & 0xFFFF0000u) * f);
    tile[u] = x;
  }
}

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;                       // [2]
  uint64_t* kv_full = bars + 2;                  // [STAGES]
  uint64_t* kv_empty = kv_full + C::STAGES;      // [STAGES]
  uint64_t* v_ready = kv_empty + C::STAGES;      // [STAGES] V slot converted to f16
  uint64_t* s_full = v_ready + C::STAGES;        // [2]
  uint64_t* p_full = s_full + 2;                 // [2]
  uint64_t* o_full = p_full + 2;                 // [2]
  uint64_t* mma_done = o_full + 2;               // [1] all MMAs of the CTA retired
  uint64_t* pass_bar = mma_done + 1;             // [1] V range of the first pass known
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pass_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* v_mag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);  // largest |V| (bf16 bits)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int BH = sh.B * sh.H;
  const int n_pairs = (N + 2 * C::BM - 1) / (2 * C::BM);
  // Heaviest causal tiles first: the last Q pair of every head leads the grid.
  const int lin = blockIdx.x;
  const int pair = n_pairs - 1 - lin / BH;
  const int bh = lin % BH;
  const int b = bh / sh.H;
  const int q0 = pair * 2 * C::BM;
  const int hh = bh % sh.H;
  const SeqView sv = seq_view<VARLEN>(args.pk, args.kv_lens, b, N);
  const int klim = sv.Lk;
  // TMA coordinates (y, z) of query row / key row `row` of this sequence.
  constexpr bool packed = VARLEN;
  auto q_yz = [&](int row, int& y, int& z) {
    y = packed ? hh : row;
    z = packed ? sv.q_start + row : bh;
  };
  auto k_yz = [&](int row, int& y, int& z) {
    y = packed ? hh : row;
    z = packed ? sv.k_start + row : bh;
  };

  // Number of key blocks each Q tile visits (fully masked blocks are skipped).
  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rs = q0 + t * C::BM;
    int kmax = klim;
    if (CAUSAL) kmax = min(kmax, rs + C::BM + sv.shift);  // last row of the tile sees keys < this
    n_t[t] = (rs >= sv.Lq || kmax <= 0) ? 0 : (kmax + C::BN - 1) / C::BN;
  }
  const int n_max = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NUM_BARS; ++i) mbar_init(&bars[i], 1);
    mbar_init(&p_full[0], 128);
    mbar_init(&p_full[1], 128);
    for (int i = 0; i < C::STAGES; ++i) mbar_init(&v_ready[i], C::CONV_THREADS);
    mbar_init(pass_bar, C::CONV_THREADS / 32);  // lane 0 of each converter warp
    *abort_flag = 0;
    *v_mag = 0;
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && !g_test_drop_loads) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (n_t[t] > 0) {
          mbar_arrive_expect_tx(&q_full[t], C::Q_BYTES);
          int y, z;
          q_yz(q0 + t * C::BM, y, z);
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_3d(smem + C::OFF_Q + t * C::Q_BYTES + c * C::SUB_BYTES, &tmQ, &q_full[t], c * 64, y, z);
        }
      }
      // One pass loads K_0, V_0, K_1, V_1, ...; ring positions count on
      // across the passes.
      const int total = 2 * n_max;
      auto load_pass = [&](int g0) {
        for (int idx = 0; idx < total; ++idx) {
          const int g = g0 + idx;
          const int slot = g % C::STAGES;
          const int use = g / C::STAGES;
          if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) return false;
          mbar_arrive_expect_tx(&kv_full[slot], C::KV_BYTES);
          const CUtensorMap* tm = (idx & 1) ? &tmV : &tmK;
          uint8_t* dst = smem + C::OFF_KV + slot * C::KV_BYTES;
          int y, z;
          k_yz((idx >> 1) * C::BN, y, z);
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_3d(dst + c * C::SUB_BYTES, tm, &kv_full[slot], c * 64, y, z);
        }
        return true;
      };
      int loads = total;
      if (load_pass(0) && n_max > 0 && mbar_wait(pass_bar, 0, abort_flag) &&
          v_second_pass_shift(*v_mag, n_max) != kNoSecondPass) {
        load_pass(total);
        loads = 2 * total;
      }
      // Do not leave with copies in flight (matters only after an abort).
      for (int g = max(0, loads - C::STAGES); g < loads; ++g)
        mbar_wait(&kv_full[g % C::STAGES], (g / C::STAGES) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0 && n_max > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t IDESC_PV = idesc_f16_f32(128, D, false, true);        // first pass: f16 P, V
      constexpr uint32_t IDESC_PV_BF16 = idesc_bf16_f32(128, D, false, true);  // second pass: bf16 P, V
      const uint32_t sbase = smem_u32(smem);
      // Operand descriptors are built once; a ring slot, a Q tile or a k-step
      // only advances the start address (sdesc_advance).
      const uint64_t dq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);             // K-major
      const uint64_t dk0 = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);            // K-major
      const uint64_t dv0 = sdesc_sw128(sbase + C::OFF_KV, C::SUB_BYTES, 1024);  // MN-major
      auto slot_bytes = [](int idx) { return static_cast<uint32_t>((idx % C::STAGES) * C::KV_BYTES); };
      auto full_wait = [&](int idx) {
        return mbar_wait(&kv_full[idx % C::STAGES], (idx / C::STAGES) & 1, abort_flag);
      };
      // S_t = Q_t K^T over D/16 k-steps (both operands K-major, 128B swizzle).
      auto issue_qk = [&](int t, int idx) {
        const uint64_t dq = sdesc_advance(dq0, t * C::Q_BYTES);
        const uint64_t dk = sdesc_advance(dk0, slot_bytes(idx));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
          tc_mma_ss(tmem + t * 128, sdesc_advance(dq, off), sdesc_advance(dk, off), IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      // O_t (+)= P_t V over 128/16 k-steps (P from TMEM over S_t, V MN-major).
      auto issue_pv = [&](int t, int idx, bool acc, uint32_t idesc) {
        const uint64_t dv = sdesc_advance(dv0, slot_bytes(idx));
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          tc_mma_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_advance(dv, kk * 16 * 128), idesc,
                    (acc || kk > 0) ? 1u : 0u);
        }
      };
      // One pass over the key blocks. Ring positions start at g0 (K_0 of the
      // pass); the per-tile barriers s_full / p_full complete n_t[t] phases
      // per pass and o_full one.
      auto run_pass = [&](int pass, uint32_t idesc_pv) {
        const int g0 = pass * 2 * n_max;
        bool ok = full_wait(g0);
        tc_fence_after();
        if (!ok) return false;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) {
            issue_qk(t, g0);
            tc_commit(&s_full[t]);
          }
        tc_commit(&kv_empty[g0 % C::STAGES]);
        for (int j = 0; j < n_max && ok; ++j) {
          const int iv = g0 + 2 * j + 1, ik = g0 + 2 * j + 2;
          ok = mbar_wait(&v_ready[iv % C::STAGES], (iv / C::STAGES) & 1, abort_flag);
          tc_fence_after();
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j < n_t[t]) {
              ok = ok && mbar_wait(&p_full[t], (pass * n_t[t] + j) & 1, abort_flag);
              tc_fence_after();
              issue_pv(t, iv, j > 0, idesc_pv);
              if (j == n_t[t] - 1) tc_commit(&o_full[t]);
            }
            if (j + 1 < n_t[t]) {
              if (!k_ready) {
                ok = ok && full_wait(ik);
                tc_fence_after();
                k_ready = true;
              }
              issue_qk(t, ik);
              tc_commit(&s_full[t]);
            }
          }
          if (j + 1 < n_max) tc_commit(&kv_empty[ik % C::STAGES]);
          tc_commit(&kv_empty[iv % C::STAGES]);
        }
        return ok;
      };
      bool ok = true;
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (n_t[t] > 0) ok = ok && mbar_wait(&q_full[t], 0, abort_flag);
      if (ok && run_pass(0, IDESC_PV) && mbar_wait(pass_bar, 0, abort_flag) &&
          v_second_pass_shift(*v_mag, n_max) != kNoSecondPass)
        run_pass(1, IDESC_PV_BF16);
      // TMEM is freed at the end: make sure no MMA is still running then.
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag);
    }
  } else if (warp < 4) {
    // ------------------------------------------------- V bf16 -> f16 in SMEM (warps 2-3)
    const int ct = threadIdx.x - 32 * C::CONV_WARP0;  // 0..CONV_THREADS-1
    float vmax = 0.f;  // largest |V| seen
    bool ok = true;
    for (int j = 0; j < n_max; ++j) {
      const int iv = 2 * j + 1;
      if (!mbar_wait(&kv_full[iv % C::STAGES], (iv / C::STAGES) & 1, abort_flag)) {
        ok = false;
        break;
      }
      uint4* tile = reinterpret_cast<uint4*>(smem + C::OFF_KV + (iv % C::STAGES) * C::KV_BYTES);
      const int rows_valid = klim - j * C::BN;  // keys of this block inside the key limit
      if (rows_valid >= C::BN)
        convert_v_f16<false, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, vmax);
      else
        convert_v_f16<true, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, vmax);
      fence_proxy_async_smem();
      mbar_arrive(&v_ready[iv % C::STAGES]);
    }
    // |V| as its bf16 bit pattern less the sign (the maximum of bf16 values
    // is a bf16 value; the order of non-negative floats is that of their bits)
    const uint32_t e = __reduce_max_sync(0xffffffffu, __float_as_uint(vmax) >> 16);
    if (lane == 0) {
      atomicMax(const_cast<uint32_t*>(v_mag), e);
      mbar_arrive(pass_bar);
    }
    // Second pass (rare): V scaled by 2^k, kept in bf16.
    if (ok && n_max > 0 && mbar_wait(pass_bar, 0, abort_flag)) {
      const int k = v_second_pass_shift(*v_mag, n_max);
      if (k != kNoSecondPass) {
        const float f = exp2i(k);
        for (int j = 0; j < n_max; ++j) {
          const int iv = 2 * n_max + 2 * j + 1;
          if (!mbar_wait(&kv_full[iv % C::STAGES], (iv / C::STAGES) & 1, abort_flag)) break;
          uint4* tile = reinterpret_cast<uint4*>(smem + C::OFF_KV + (iv % C::STAGES) * C::KV_BYTES);
          const int rows_valid = klim - j * C::BN;
          if (rows_valid >= C::BN)
            scale_v_bf16<false, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, f);
          else
            scale_v_bf16<true, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, f);
          fence_proxy_async_smem();
          mbar_arrive(&v_ready[iv % C::STAGES]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 4-11)
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row_start = q0 + t * C::BM;
    const int r = row_start + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const float sl2 = sh.scale_log2;
    const int nt = n_t[t];
    float m_used = -INFINITY;  // reference max, base-2 units of scaled logits
    float l = 0.f;             // row sum of the P values (which carry the factor 2^7)
    int shift = kNoSecondPass;  // V scale exponent of the second pass, if it runs
    bool ok = true;
    for (int pass = 0; pass < 2; ++pass) {
      m_used = -INFINITY;
      l = 0.f;
      for (int j = 0; j < nt; ++j) {
        // warp-collective TMEM ops follow
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], (pass * nt + j) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
        const int kb = j * C::BN;
        const bool need_mask = (kb + C::BN > klim) || (CAUSAL && kb + C::BN - 1 > row_start + sv.shift);
        const int cmax = CAUSAL ? min(klim, r + 1 + sv.shift) : klim;  // visible keys: c < cmax
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (kb + c >= cmax) s[c] = __float_as_uint(-INFINITY);
        }
        float mx = __uint_as_float(s[0]);
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
        const float m_new = fmaxf(m_used, mx * sl2);
        const bool resc = m_new > m_used + 8.0f;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2(m_used - m_new);  // 0 on the first block (m_used = -inf)
          m_used = m_new;
        }
        l *= alpha;
        // p = 2^(s*sl2 - m_used + 7): the factor 2^7 keeps small p off f16's subnormals.
        const float msub = ((m_used == -INFINITY) ? 0.f : m_used) - 7.0f;
        float rs0 = 0.f, rs1 = 0.f;
        if (pass == 0)
          softmax_exp_store_f16(s, sl2, msub, rs0, rs1, tS);
        else
          softmax_exp_store_bf16(tS, sl2, msub, kb, cmax, rs0, rs1);
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O_t is idle here: the commit that signalled S_t(j) also covers PV(j-1),
          // and PV(j) waits for p_full below.
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_wait_st();
        l += rs0 + rs1;
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      if (nt == 0 || !ok) break;
      ok = mbar_wait(&o_full[t], pass & 1, abort_flag);
      tc_fence_after();
      if (!ok || pass == 1) break;
      // The V range of the first pass decides whether the scan repeats in bf16.
      ok = __all_sync(0xffffffffu, mbar_wait(pass_bar, 0, abort_flag));
      if (!ok) break;
      shift = v_second_pass_shift(*v_mag, n_max);
      if (shift == kNoSecondPass) break;
    }
    // ----------------------------------------------------------- epilogue
    if (row_start < sv.Lq) {  // uniform over the tile's 128 threads
      const bool valid = r < sv.Lq;
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float unscale = (shift == kNoSecondPass) ? 1.f : exp2i(-shift);  // undo V's 2^k
      // O leaves through this tile's Q buffer, idle now (every product that
      // read it has completed): each thread writes its row there in the
      // 128B-swizzled layout (conflict-free: 8 consecutive rows cover all
      // banks), then the tile's threads copy the buffer out in whole 128-byte
      // row segments, where one 16-byte store per thread would touch 32 rows
      // per warp instruction.
      fence_proxy_async_smem();  // the products' reads of Q before these writes
      uint8_t* stage = smem + C::OFF_Q + t * C::Q_BYTES;
      const int rt = wq * 32 + lane;  // row within the tile
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv * unscale, __uint_as_float(o[2 * i + 1]) * inv * unscale);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const int u8 = (c & 1) * 4 + v4;  // 16-byte unit within the 64-column chunk c / 2
          *reinterpret_cast<uint4*>(stage + (c >> 1) * C::SUB_BYTES + rt * 128 + ((u8 ^ (rt & 7)) << 4)) =
              make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
      }
      named_bar_sync(1 + t, 128);
      // Output rows of this sequence: [B,H,N,d] or packed [total,H,d].
      constexpr int UPR = D / 8;  // 16-byte units per row
#pragma unroll 4
      for (int f = rt; f < C::BM * UPR; f += 128) {
        const int row = f / UPR, uu = f % UPR;
        if (row_start + row < sv.Lq) {
          const uint4 x = *reinterpret_cast<const uint4*>(stage + (uu >> 3) * C::SUB_BYTES + row * 128 +
                                                          (((uu & 7) ^ (row & 7)) << 4));
          reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) +
                                   q_row<VARLEN>(args.pk, sh, sv, bh, row_start + row) * D)[uu] = x;
        }
      }
      // LSE [B,H,N] or [H,total]: one float per row, consecutive across the warp.
      if (valid)
        args.lse[lse_index<VARLEN>(args.pk, sh, sv, bh, r)] = (l > 0.f) ? (m_used + log2f(l) - 7.0f) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

cudaError_t set_fwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_fwd_status() { return take_status_here(); }

template <int D, bool CAUSAL, bool VARLEN>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdArgs& a, cudaStream_t stream, const LaunchMarks* marks) {
  using C = FwdCfg<D>;
  auto kern = fa_fwd_kernel<D, CAUSAL, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int BH = a.s.B * a.s.H;
  const int n_pairs = (a.s.N + 2 * C::BM - 1) / (2 * C::BM);
  const long long blocks = static_cast<long long>(n_pairs) * BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  mark(marks, true, 0, stream);
  kern<<<static_cast<unsigned>(blocks), C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, a);
  mark(marks, false, 0, stream);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                       cudaStream_t stream, const LaunchMarks* m) {
  const bool c = a.s.causal != 0;
  if (a.pk.varlen) {
    if (a.s.D == 64)
      return c ? launch_fwd_t<64, true, true>(tq, tk, tv, a, stream, m)
               : launch_fwd_t<64, false, true>(tq, tk, tv, a, stream, m);
    return c ? launch_fwd_t<128, true, true>(tq, tk, tv, a, stream, m)
             : launch_fwd_t<128, false, true>(tq, tk, tv, a, stream, m);
  }
  if (a.s.D == 64)
    return c ? launch_fwd_t<64, true, false>(tq, tk, tv, a, stream, m)
             : launch_fwd_t<64, false, false>(tq, tk, tv, a, stream, m);
  return c ? launch_fwd_t<128, true, false>(tq, tk, tv, a, stream, m)
           : launch_fwd_t<128, false, false>(tq, tk, tv, a, stream, m);
}

}  // namespace fa
