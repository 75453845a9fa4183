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
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: one thread per
//               query row (TMEM lane), exp2-domain online softmax, P written
//               back to TMEM as f16, O rescaled in TMEM only when the running
//               max grows by more than 2^8 (exact: m, l and O share the same
//               reference max), then the epilogue O = acc / l and LSE.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
//
// Range of V. f16 holds bf16 values exactly only for magnitudes in
// [2^-14, 65536): a larger |V| becomes inf in f16, a smaller one lands on
// f16's subnormal grid (absolute error 2^-25). The first pass runs P V in f16
// for every tile; the epilogue then checks each row of O, which costs nothing
// per key block: a non-finite O (an f16 overflow, or inf/NaN input) or a row
// whose largest |O| is below 2^-16 (V this small loses relative precision)
// flags the Q tile. A flagged tile (rare) is computed again: the converter
// warps first find the exact largest |V| over the CTA's visible keys (a scan
// of the V tiles, loaded once more), then the tile's scan repeats with V
// scaled in shared memory by 2^k (exact; the largest magnitude then lies in
// [2, 4)), P quantised to bf16 (fp32's exponent range) and P V in bf16; the
// epilogue multiplies O by 2^-k. Keys at or past the key limit are zeroed in
// shared memory in every pass (padding or the next packed sequence can hold
// anything). P carries a factor 2^7 (in the exponent; l carries it too, so O =
// acc / l is unchanged and the LSE subtracts 7): with the lazy rescale P stays
// below 2^15, inside f16's range, and probabilities down to 2^-38 of the
// running maximum keep f16 normals instead of flushing to zero.
#include <algorithm>
#include <atomic>

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
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16 + 1024;  // + 4 words, alignment slack
  static constexpr int THREADS = 384;
  static constexpr int CONV_WARP0 = 2;     // warps 2-3 convert V
  static constexpr int CONV_THREADS = 64;
  static constexpr uint32_t TMEM_COLS = 512;
};

// Power-of-two shift k of V for the bf16 pass, from the largest bf16
// magnitude (the 15 bits below the sign) among the V values of the keys the
// CTA sees: with e the largest exponent field, k = 128 - e puts the largest
// magnitude in [2, 4); k is capped at 126 (V made only of bf16 subnormals) so
// that 2^k and 2^-k stay normal fp32 numbers. An all-zero V and non-finite
// values keep k = 0 (O stays 0, or non-finite as the definition gives).
__device__ __forceinline__ int v_scale_shift(uint32_t vmag) {
  const int e = static_cast<int>(vmag >> 7);
  if (vmag == 0 || e == 255) return 0;
  return min(128 - e, 126);
}

// max(a, |b|, |c|), NaN if any operand is NaN (one instruction).
__device__ __forceinline__ float max3_nan_abs(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

// A row of the first pass needs the bf16 pass when its O holds inf or NaN,
// or when every |O| of a row with visible keys is below 2^-16 (then V is so
// small that f16's subnormal grid matters). ``omax`` is the largest |O| of
// the row (NaN if any element is NaN).
__device__ __forceinline__ bool row_needs_bf16_pass(float omax, float l) {
  return !(omax <= 3.0e38f) || (l > 0.f && omax < 1.52587890625e-5f);
}

// 2^e as an fp32 constant, for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// Largest logit of the row (masked keys excluded), read from TMEM in two
// 64-column halves so that only half a row is held in registers.
__device__ __forceinline__ float softmax_row_max(uint32_t tS, bool need_mask, int kb, int cmax) {
  if (!need_mask) {
    // No masked key in the block: the TMEM loads reduce the row themselves.
    uint32_t s[64];
    float m0, m1;
    tmem_ld64_max(tS, s, m0);
    tmem_wait_ld();
    tmem_ld64_max(tS + 64, s, m1);
    tmem_wait_ld();
    return fmaxf(m0, m1);
  }
  float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t s[64];
    tmem_ld32(tS + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_ld32(tS + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_wait_ld();
    if (need_mask) {
#pragma unroll
      for (int cc = 0; cc < 64; ++cc)
        if (kb + hh * 64 + cc >= cmax) s[cc] = __float_as_uint(-INFINITY);
    }
    // four independent chains of 3-input maxima
#pragma unroll
    for (int cc = 0; cc < 64; cc += 8) {
#pragma unroll
      for (int q = 0; q < 4; ++q) mq[q] = max3f(mq[q], __uint_as_float(s[cc + 2 * q]), __uint_as_float(s[cc + 2 * q + 1]));
    }
  }
  return fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
}

// p = 2^(s * sl2 - msub) for the 128 logits of the row, re-read from TMEM a
// half at a time, summed into rs0 / rs1 and written back over S as 64 packed
// f16 pairs (bf16 in the second pass; half hh of P lands on columns
// [32 hh, 32 hh + 32), which hold logits already read). The scaling and the
// sums run two lanes per instruction (f32x2); both passes add in the same
// order, so a row gets the same sum, and LSE, from either.
template <bool BF16>
__device__ __forceinline__ void softmax_exp_store(uint32_t tS, bool need_mask, int kb, int cmax, float sl2,
                                                  float msub, float& rs0, float& rs1) {
  const uint64_t scale2 = f2_pack(sl2, sl2), neg2 = f2_pack(-msub, -msub);
  uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t s[64];
    tmem_ld32(tS + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_ld32(tS + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_wait_ld();
    if (need_mask) {
#pragma unroll
      for (int cc = 0; cc < 64; ++cc)
        if (kb + hh * 64 + cc >= cmax) s[cc] = __float_as_uint(-INFINITY);
    }
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), scale2, neg2);
      float x0, x1;
      f2_unpack(x, x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      acc[i & 1] = f2_add(acc[i & 1], f2_pack(p0, p1));
      pk[i] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
    }
    tmem_st32(tS + hh * 32, pk);
  }
  float a0, a1, b0, b1;
  f2_unpack(acc[0], a0, a1);
  f2_unpack(acc[1], b0, b1);
  rs0 += a0 + b0;
  rs1 += a1 + b1;
}

// exp2 of one 64-column half already in registers (same arithmetic and sum
// order as softmax_exp_store), P stored over columns [32 hh, 32 hh + 32).
template <bool BF16>
__device__ __forceinline__ void softmax_exp_half(const uint32_t (&s)[64], uint64_t scale2, uint64_t neg2,
                                                 uint64_t (&acc)[2], uint32_t tS, int hh) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), scale2, neg2);
    float x0, x1;
    f2_unpack(x, x0, x1);
    const float p0 = ex2(x0), p1 = ex2(x1);
    acc[i & 1] = f2_add(acc[i & 1], f2_pack(p0, p1));
    pk[i] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
  }
  tmem_st32(tS + hh * 32, pk);
}

// The dynamic shared memory of the forward kernel (1024-byte aligned by the
// user of this pointer).
__device__ __forceinline__ uint8_t* fwd_smem_base() {
  extern __shared__ uint8_t fwd_smem_raw[];
  return fwd_smem_raw;
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

// First pass: bf16 -> f16 in place.
template <bool MASK, int UNITS, int CT>
__device__ __forceinline__ void convert_v_f16(uint4* tile, int rows_valid, int ct) {
#pragma unroll 4
  for (int u = ct; u < UNITS; u += CT) {
    uint4 x = load_v_unit<MASK>(tile, u, rows_valid);
    x.x = bf16x2_to_f16x2(x.x);
    x.y = bf16x2_to_f16x2(x.y);
    x.z = bf16x2_to_f16x2(x.z);
    x.w = bf16x2_to_f16x2(x.w);
    tile[u] = x;
  }
}

// Range scan (rare path): the largest bf16 magnitude per 16-bit half of the
// tile's visible keys, folded into ``vmag``.
template <bool MASK, int UNITS, int CT>
__device__ __forceinline__ void scan_v_mag(const uint4* tile, int rows_valid, int ct, uint32_t& vmag) {
  for (int u = ct; u < UNITS; u += CT) {
    const uint4 x = load_v_unit<MASK>(tile, u, rows_valid);
    vmag = __vimax3_u16x2(vmag, x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu);
    vmag = __vimax3_u16x2(vmag, x.z & 0x7FFF7FFFu, x.w & 0x7FFF7FFFu);
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

// ---------------------------------------------------------------------------
// Shared-memory layout of one CTA and the per-role steps, used by the kernel
// for the f16 pass and by the (rare) bf16 pass.
// ---------------------------------------------------------------------------
template <int D>
struct FwdShared {
  uint8_t* smem;
  uint64_t *q_full, *kv_full, *kv_empty, *v_ready, *s_full, *p_full, *o_full, *mma_done, *scan_done;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile uint32_t* redo;   // bit t: tile t takes the bf16 pass
  volatile uint32_t* v_mag;  // largest |V| (bf16 bits) of the range scan
  __device__ explicit FwdShared(uint8_t* base) : smem(base) {
    using C = FwdCfg<D>;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    q_full = bars;                   // [2]
    kv_full = bars + 2;              // [STAGES]
    kv_empty = kv_full + C::STAGES;  // [STAGES]
    v_ready = kv_empty + C::STAGES;  // [STAGES] V slot converted (f16, or scaled bf16)
    s_full = v_ready + C::STAGES;    // [2]
    p_full = s_full + 2;             // [2]
    o_full = p_full + 2;             // [2]
    mma_done = o_full + 2;           // [1] all MMAs issued so far retired
    scan_done = mma_done + 1;        // [1] largest |V| known (bf16 pass)
    tmem_slot = reinterpret_cast<uint32_t*>(scan_done + 1);
    abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    redo = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
    v_mag = reinterpret_cast<volatile uint32_t*>(tmem_slot + 3);
  }
};

// What one CTA works on: two 128-row Q tiles of one (b, h).
struct FwdCta {
  int q0, bh, hh, klim, n_max;
  int own;     // bit t: this CTA computes and writes tile t (both, unless the pair is split)
  int n_t[2];  // key blocks each Q tile visits (fully masked blocks are skipped)
  SeqView sv;
  uint32_t tmem;
};

template <int D, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdCta fwd_cta(const FwdArgs& args) {
  using C = FwdCfg<D>;
  const AttnShape& sh = args.s;
  const int BH = sh.B * sh.H;
  const int n_pairs = (sh.N + 2 * C::BM - 1) / (2 * C::BM);
  // The grid runs in groups of heads whose K and V fit the L2 together (every
  // Q pair of a head reads all of its K and V), and inside a group heaviest
  // causal tiles first: the last Q pair of every head of the group leads.
  // The last pairs of the grid order may run as two single-tile CTAs (the
  // launch adds one CTA per split pair): pairs [2 P - grid, P).
  const int P = BH * n_pairs;
  const int split_from = 2 * P - static_cast<int>(gridDim.x);
  int lin = blockIdx.x;
  int own = 3;
  if (lin >= split_from) {
    const int sidx = lin - split_from;
    lin = split_from + (sidx >> 1);
    own = 1 << (sidx & 1);
  }
  const int G = min(BH, max(1, args.heads_per_group));
  const int group = lin / (G * n_pairs);
  const int gsize = min(G, BH - group * G);
  const int r_in = lin - group * G * n_pairs;
  const int pair = n_pairs - 1 - r_in / gsize;
  FwdCta c;
  c.bh = group * G + r_in % gsize;
  c.hh = c.bh % sh.H;
  c.q0 = pair * 2 * C::BM;
  c.sv = seq_view<VARLEN>(args.pk, args.kv_lens, c.bh / sh.H, sh.N);
  c.klim = c.sv.Lk;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rs = c.q0 + t * C::BM;
    int kmax = c.klim;
    if (CAUSAL) kmax = min(kmax, rs + C::BM + c.sv.shift);  // last row of the tile sees keys < this
    c.n_t[t] = (rs >= c.sv.Lq || kmax <= 0 || !((own >> t) & 1)) ? 0 : (kmax + C::BN - 1) / C::BN;
  }
  c.own = own;
  c.n_max = max(c.n_t[0], c.n_t[1]);
  return c;
}

// TMA: ring positions g0 + i0 .. g0 + i1 - 1 (even offsets K_(i/2), odd
// offsets V_(i/2)); each slot is reused once its consumers have released it.
// Returns the ring position after the last load issued (g0 + i1 unless a wait
// gave up).
template <int D, bool VARLEN>
__device__ __forceinline__ int fwd_load_kv_range(const FwdShared<D>& sm, const FwdCta& c, const CUtensorMap* tmK,
                                                 const CUtensorMap* tmV, int g0, int i0, int i1) {
  using C = FwdCfg<D>;
  for (int idx = i0; idx < i1; ++idx) {
    const int g = g0 + idx;
    const int slot = g % C::STAGES;
    const int use = g / C::STAGES;
    if (use > 0 && !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, sm.abort_flag)) return g;
    mbar_arrive_expect_tx(&sm.kv_full[slot], C::KV_BYTES);
    const CUtensorMap* tm = (idx & 1) ? tmV : tmK;
    uint8_t* dst = sm.smem + C::OFF_KV + slot * C::KV_BYTES;
    const int row = (idx >> 1) * C::BN;
    const int y = VARLEN ? c.hh : row;
    const int z = VARLEN ? c.sv.k_start + row : c.bh;
#pragma unroll
    for (int cc = 0; cc < C::CHUNKS; ++cc) tma_load_3d(dst + cc * C::SUB_BYTES, tm, &sm.kv_full[slot], cc * 64, y, z);
  }
  return g0 + i1;
}

// TMA: K_0, V_0, K_1, V_1, ... of n key blocks into ring positions g0, g0+1,
// ... Returns the ring position after the last load issued (g0 + 2 n unless a
// wait gave up).
template <int D, bool VARLEN>
__device__ __forceinline__ int fwd_load_kv(const FwdShared<D>& sm, const FwdCta& c, const CUtensorMap* tmK,
                                           const CUtensorMap* tmV, int g0, int n) {
  return fwd_load_kv_range<D, VARLEN>(sm, c, tmK, tmV, g0, 0, 2 * n);
}

// Wait for the ring copies in flight, the last STAGES positions before
// ``loads`` (every one of them issued). Matters only after an abort, when the
// consumers stopped waiting; every issued copy still lands, so the bound is
// not reached.
template <int D>
__device__ __forceinline__ void fwd_drain_loads(const FwdShared<D>& sm, int loads) {
  using C = FwdCfg<D>;
  for (int g = max(0, loads - C::STAGES); g < loads; ++g)
    mbar_wait_drain(&sm.kv_full[g % C::STAGES], (g / C::STAGES) & 1);
}

// MMA warp (all lanes run the loop, one elected lane issues): one pass over
// the key blocks. Tile t visits nb[t]
// blocks; its barriers s_full / p_full have completed base[t] phases before
// the pass; ring positions start at g0 (K_0 of the pass).
template <int D>
__device__ __forceinline__ bool fwd_mma_pass(const FwdShared<D>& sm, uint32_t tmem, const int (&nb)[2],
                                             const int (&base)[2], int g0, uint32_t idesc_pv) {
  using C = FwdCfg<D>;
  constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);
  const uint32_t sbase = smem_u32(sm.smem);
  // Operand descriptors are built once; a ring slot, a Q tile or a k-step
  // only advances the start address (sdesc_advance).
  const uint64_t dq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);             // K-major
  const uint64_t dk0 = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);            // K-major
  const uint64_t dv0 = sdesc_sw128(sbase + C::OFF_KV, C::SUB_BYTES, 1024);  // MN-major
  auto slot_bytes = [](int idx) { return static_cast<uint32_t>((idx % C::STAGES) * C::KV_BYTES); };
  auto full_wait = [&](int idx) {
    return __all_sync(0xffffffffu, mbar_wait(&sm.kv_full[idx % C::STAGES], (idx / C::STAGES) & 1, sm.abort_flag));
  };
  // S_t = Q_t K^T over D/16 k-steps (both operands K-major, 128B swizzle).
  auto issue_qk = [&](int t, int idx) {
    const uint64_t dq = sdesc_advance(dq0, t * C::Q_BYTES);
    const uint64_t dk = sdesc_advance(dk0, slot_bytes(idx));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
      tc_mma_ss_w(tmem + t * 128, sdesc_advance(dq, off), sdesc_advance(dk, off), IDESC_QK, kk > 0 ? 1u : 0u);
    }
  };
  // O_t (+)= P_t V over 128/16 k-steps (P from TMEM over S_t, V MN-major).
  auto issue_pv = [&](int t, int idx, bool acc) {
    const uint64_t dv = sdesc_advance(dv0, slot_bytes(idx));
#pragma unroll
    for (int kk = 0; kk < C::BN / 16; ++kk) {
      tc_mma_ts_w(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_advance(dv, kk * 16 * 128), idesc_pv,
                  (acc || kk > 0) ? 1u : 0u);
    }
  };
  const int nmax = max(nb[0], nb[1]);
  bool ok = full_wait(g0);
  tc_fence_after();
  if (!ok) return false;
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (nb[t] > 0) {
      // Q_t (its load completes phase 0 of q_full[t]; a later pass finds it done)
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_full[t], 0, sm.abort_flag))) return false;
      tc_fence_after();
      issue_qk(t, g0);
      tc_commit_w(&sm.s_full[t]);
    }
  tc_commit_w(&sm.kv_empty[g0 % C::STAGES]);
  for (int j = 0; j < nmax && ok; ++j) {
    const int iv = g0 + 2 * j + 1, ik = g0 + 2 * j + 2;
    ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_ready[iv % C::STAGES], (iv / C::STAGES) & 1, sm.abort_flag));
    tc_fence_after();
    bool k_ready = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (j < nb[t]) {
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&sm.p_full[t], (base[t] + j) & 1, sm.abort_flag));
        tc_fence_after();
        issue_pv(t, iv, j > 0);
        if (j == nb[t] - 1) tc_commit_w(&sm.o_full[t]);
      }
      if (j + 1 < nb[t]) {
        if (!k_ready) {
          ok = ok && full_wait(ik);
          tc_fence_after();
          k_ready = true;
        }
        issue_qk(t, ik);
        tc_commit_w(&sm.s_full[t]);
      }
    }
    if (j + 1 < nmax) tc_commit_w(&sm.kv_empty[ik % C::STAGES]);
    tc_commit_w(&sm.kv_empty[iv % C::STAGES]);
  }
  return ok;
}

// Softmax of one Q tile (128 threads, one query row each) over nt key
// blocks: the online-softmax recurrence, P back into TMEM (f16 in the first
// pass, bf16 in the second), O rescaled lazily. Returns false if a wait gave
// up; m_used and l are the row's reference max (base 2) and sum of P.
template <int D, bool CAUSAL, bool BF16>
__device__ __forceinline__ bool fwd_softmax_pass(const FwdShared<D>& sm, const FwdCta& c, int t, int r, uint32_t tS,
                                                 uint32_t tO, float sl2, int phase0, float& m_used, float& l) {
  using C = FwdCfg<D>;
  const int nt = c.n_t[t];
  const int row_start = c.q0 + t * C::BM;
  m_used = -INFINITY;
  l = 0.f;
  for (int j = 0; j < nt; ++j) {
    // warp-collective TMEM ops follow
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], (phase0 + j) & 1, sm.abort_flag))) return false;
    tc_fence_after();
    const int kb = j * C::BN;
    const bool need_mask = (kb + C::BN > c.klim) || (CAUSAL && kb + C::BN - 1 > row_start + c.sv.shift);
    const int cmax = CAUSAL ? min(c.klim, r + 1 + c.sv.shift) : c.klim;  // visible keys: c < cmax
    bool resc = false;
    float alpha = 1.f;
    // The reference max moves only when the block's max exceeds it by more
    // than 2^8 (lazy rescale); returns the exponent offset of P.
    auto update = [&](float mx) {
      const float m_new = fmaxf(m_used, mx * sl2);
      resc = m_new > m_used + 8.0f;
      if (resc) {
        alpha = ex2(m_used - m_new);  // 0 on the first block (m_used = -inf)
        m_used = m_new;
      }
      l *= alpha;
      // p = 2^(s*sl2 - m_used + 7): the factor 2^7 keeps small p off f16's subnormals.
      return ((m_used == -INFINITY) ? 0.f : m_used) - 7.0f;
    };
    float rs0 = 0.f, rs1 = 0.f;
    if (!need_mask) {
      // No masked key: the TMEM loads reduce the row themselves, and the
      // second of them keeps half 0's logits for the exponentials.
      uint32_t s[64];
      float m0, m1;
      tmem_ld64_max(tS + 64, s, m1);
      tmem_wait_ld();
      tmem_ld64_max(tS, s, m0);
      tmem_wait_ld();
      const float msub = update(fmaxf(m0, m1));
      const uint64_t scale2 = f2_pack(sl2, sl2), neg2 = f2_pack(-msub, -msub);
      uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      softmax_exp_half<BF16>(s, scale2, neg2, acc, tS, 0);
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_wait_ld();
      softmax_exp_half<BF16>(s, scale2, neg2, acc, tS, 1);
      float a0, a1, b0, b1;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], b0, b1);
      rs0 += a0 + b0;
      rs1 += a1 + b1;
    } else {
      const float msub = update(softmax_row_max(tS, need_mask, kb, cmax));
      softmax_exp_store<BF16>(tS, need_mask, kb, cmax, sl2, msub, rs0, rs1);
    }
    if (j > 0 && __any_sync(0xffffffffu, resc)) {
      // O_t is idle here: the commit that signalled S_t(j) also covers PV(j-1),
      // and PV(j) waits for p_full below.
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + cc * 32, o);
      }
    }
    tmem_wait_st();
    l += rs0 + rs1;
    tc_fence_before();
    mbar_arrive(&sm.p_full[t]);
  }
  return true;
}

// Epilogue of one row: O = acc / l (times ``unscale``) as bf16 and LSE.
// Returns the row's largest |O| (NaN if an element is NaN).
template <int D, bool VARLEN>
__device__ __forceinline__ float fwd_epilogue(const FwdArgs& args, const FwdCta& c, int r, uint32_t tO, bool have_o,
                                              float m_used, float l, float unscale) {
  const bool valid = r < c.sv.Lq;
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  // Output row r of this sequence: [B,H,N,d] or packed [total,H,d]; LSE
  // [B,H,N] or [H,total].
  uint4* orow =
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + q_row<VARLEN>(args.pk, args.s, c.sv, c.bh, r) * D);
  float omax = 0.f;
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(tO + cc * 32, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0u;
    }
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float a0 = __uint_as_float(o[2 * i]) * inv * unscale;
      const float a1 = __uint_as_float(o[2 * i + 1]) * inv * unscale;
      omax = max3_nan_abs(omax, a0, a1);
      w[i] = pack_bf16x2(a0, a1);
    }
    if (valid) {
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4)
        orow[cc * 4 + v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
    }
  }
  if (valid)
    args.lse[lse_index<VARLEN>(args.pk, args.s, c.sv, c.bh, r)] =
        (l > 0.f) ? (m_used + log2f(l) - 7.0f) * kLn2 : -INFINITY;
  return omax;
}

// ---------------------------------------------------------------------------
// bf16 pass of the Q tiles flagged in *redo, run by every thread of the CTA
// after the first pass (rarely: V outside f16's exact range). Out of line, so
// that the first pass's code does not carry it. Ring positions [2 n_max,
// 2 n_max + 2 n_r) carry the range scan (the converters read V; the K loads
// keep K and V in their usual slots and are not read), [2 n_max + 2 n_r,
// + 2 n_r) the pass itself; every barrier continues from its first-pass phase.
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL, bool VARLEN>
__device__ __noinline__ void fwd_bf16_pass(const CUtensorMap* tmK, const CUtensorMap* tmV, FwdArgs args, FwdCta c,
                                           uint32_t mask) {
  using C = FwdCfg<D>;
  const FwdShared<D> sm(reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(fwd_smem_base()) + 1023) & ~uintptr_t(1023)));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb2[2] = {(mask & 1u) ? c.n_t[0] : 0, (mask & 2u) ? c.n_t[1] : 0};
  const int n_r = max(nb2[0], nb2[1]);
  const int g_scan = 2 * c.n_max, g_pass = g_scan + 2 * n_r;
  if (warp == 0) {
    if (lane == 0 && !g_test_drop_loads) {
      int loads = fwd_load_kv<D, VARLEN>(sm, c, tmK, tmV, g_scan, n_r);
      if (loads == g_pass) loads = fwd_load_kv<D, VARLEN>(sm, c, tmK, tmV, g_pass, n_r);
      fwd_drain_loads<D>(sm, loads);
    }
  } else if (warp == 1) {
    // Every ring position of the scan (which the MMA warp skips) has
    // completed once scan_done has: the parity waits below cannot alias.
    if (__all_sync(0xffffffffu, mbar_wait(sm.scan_done, 0, sm.abort_flag)))
      fwd_mma_pass<D>(sm, c.tmem, nb2, c.n_t, g_pass, idesc_bf16_f32(128, D, false, true));
    tc_commit_w(sm.mma_done);
    mbar_wait_drain(sm.mma_done, 1);
  } else if (warp < 4) {
    const int ct = threadIdx.x - 32 * C::CONV_WARP0;
    bool ok = true;
    uint32_t vmag = 0;
    for (int j = 0; j < n_r && ok; ++j) {
      const int ik = g_scan + 2 * j, iv = ik + 1;
      ok = mbar_wait(&sm.kv_full[ik % C::STAGES], (ik / C::STAGES) & 1, sm.abort_flag) &&
           mbar_wait(&sm.kv_full[iv % C::STAGES], (iv / C::STAGES) & 1, sm.abort_flag);
      if (ok) {
        const uint4* tile = reinterpret_cast<const uint4*>(sm.smem + C::OFF_KV + (iv % C::STAGES) * C::KV_BYTES);
        const int rows_valid = c.klim - j * C::BN;
        if (rows_valid >= C::BN)
          scan_v_mag<false, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, vmag);
        else
          scan_v_mag<true, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, vmag);
      }
      // Complete the V slot's conversion phase (as every V load in that slot
      // does), then, once both converter warps have read the slot and
      // arrived, release the V slot and the (unread) K slot.
      mbar_arrive(&sm.v_ready[iv % C::STAGES]);
      ok = named_bar_and(3, C::CONV_THREADS, ok);
      if (ct == 0) {
        mbar_arrive(&sm.kv_empty[ik % C::STAGES]);
        mbar_arrive(&sm.kv_empty[iv % C::STAGES]);
      }
    }
    const uint32_t e = __reduce_max_sync(0xffffffffu, max(vmag & 0xFFFFu, vmag >> 16));
    if (lane == 0) {
      atomicMax(const_cast<uint32_t*>(sm.v_mag), e);
      mbar_arrive(sm.scan_done);
    }
    if (ok && mbar_wait(sm.scan_done, 0, sm.abort_flag)) {
      const float f = exp2i(v_scale_shift(*sm.v_mag));
      for (int j = 0; j < n_r; ++j) {
        const int iv = g_pass + 2 * j + 1;
        if (!mbar_wait(&sm.kv_full[iv % C::STAGES], (iv / C::STAGES) & 1, sm.abort_flag)) break;
        uint4* tile = reinterpret_cast<uint4*>(sm.smem + C::OFF_KV + (iv % C::STAGES) * C::KV_BYTES);
        const int rows_valid = c.klim - j * C::BN;
        if (rows_valid >= C::BN)
          scale_v_bf16<false, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, f);
        else
          scale_v_bf16<true, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct, f);
        fence_proxy_async_smem();
        mbar_arrive(&sm.v_ready[iv % C::STAGES]);
      }
    }
  } else {
    const int t = (warp - 4) >> 2;
    if (!((mask >> t) & 1u)) return;
    const int wq = warp & 3;
    const int r = c.q0 + t * C::BM + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = c.tmem + lane_off + t * 128;
    const uint32_t tO = c.tmem + lane_off + 256 + t * D;
    float m_used, l;
    bool ok = fwd_softmax_pass<D, CAUSAL, true>(sm, c, t, r, tS, tO, args.s.scale_log2, c.n_t[t], m_used, l);
    ok = ok && mbar_wait(&sm.o_full[t], 1, sm.abort_flag);
    tc_fence_after();
    ok = ok && mbar_wait(sm.scan_done, 0, sm.abort_flag);
    // V was scaled by 2^k: O comes back by 2^-k.
    fwd_epilogue<D, VARLEN>(args, c, r, tO, true, m_used, l, ok ? exp2i(-v_scale_shift(*sm.v_mag)) : 1.f);
  }
}

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D>;
  const FwdShared<D> sm(reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(fwd_smem_base()) + 1023) & ~uintptr_t(1023)));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  FwdCta c = fwd_cta<D, CAUSAL, VARLEN>(args);
  // Packed batches size the grid by the longest sequence: a CTA whose tiles
  // lie past the end of its sequence has nothing to write and leaves before
  // any set-up (the whole CTA takes this branch).
  if (VARLEN && !((c.own & 1) && c.q0 < c.sv.Lq) && !((c.own & 2) && c.q0 + C::BM < c.sv.Lq)) return;

  // Thread 0 (the TMA thread) first initialises the barriers the first
  // copies complete on and issues Q_0, K_0, Q_1 and V_0, so that their
  // latency overlaps the rest of the set-up.
  auto load_q = [&](int t) {
    if (c.n_t[t] > 0) {
      mbar_arrive_expect_tx(&sm.q_full[t], C::Q_BYTES);
      const int row = c.q0 + t * C::BM;
      const int y = VARLEN ? c.hh : row;
      const int z = VARLEN ? c.sv.q_start + row : c.bh;
#pragma unroll
      for (int cc = 0; cc < C::CHUNKS; ++cc)
        tma_load_3d(sm.smem + C::OFF_Q + t * C::Q_BYTES + cc * C::SUB_BYTES, &tmQ, &sm.q_full[t], cc * 64, y, z);
    }
  };
  const int early = min(2, 2 * c.n_max);  // ring positions issued in the set-up
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) mbar_init(&sm.q_full[t], 1);
    for (int i = 0; i < C::STAGES; ++i) mbar_init(&sm.kv_full[i], 1);
    fence_mbar_init();
    if (!g_test_drop_loads) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      load_q(0);
      fwd_load_kv_range<D, VARLEN>(sm, c, &tmK, &tmV, 0, 0, min(1, early));
      load_q(1);
      fwd_load_kv_range<D, VARLEN>(sm, c, &tmK, &tmV, 0, min(1, early), early);
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm.smem + C::OFF_BAR);
    for (int i = 2 + C::STAGES; i < C::NUM_BARS; ++i) mbar_init(&bars[i], 1);  // after q_full, kv_full
    mbar_init(&sm.p_full[0], 128);
    mbar_init(&sm.p_full[1], 128);
    for (int i = 0; i < C::STAGES; ++i) mbar_init(&sm.v_ready[i], C::CONV_THREADS);
    mbar_init(sm.scan_done, C::CONV_THREADS / 32);  // lane 0 of each converter warp
    *sm.abort_flag = 0;
    *sm.redo = 0;
    *sm.v_mag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *sm.tmem_slot;
  // A backward pre-pass launched programmatically after this kernel may start
  // once every CTA of this grid is running (it waits for this grid to finish
  // before it reads O and LSE).
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && !g_test_drop_loads) {
      fwd_drain_loads<D>(sm, fwd_load_kv_range<D, VARLEN>(sm, c, &tmK, &tmV, 0, early, 2 * c.n_max));
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (c.n_t[t] > 0) mbar_wait_drain(&sm.q_full[t], 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (c.n_max > 0) {
      const int zero[2] = {0, 0};
      fwd_mma_pass<D>(sm, c.tmem, c.n_t, zero, 0, idesc_f16_f32(128, D, false, true));
      // TMEM is freed at the end: make sure no MMA is still running then.
      tc_commit_w(sm.mma_done);
      mbar_wait_drain(sm.mma_done, 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------- V bf16 -> f16 in SMEM (warps 2-3)
    const int ct = threadIdx.x - 32 * C::CONV_WARP0;  // 0..CONV_THREADS-1
    for (int j = 0; j < c.n_max; ++j) {
      const int iv = 2 * j + 1;
      if (!mbar_wait(&sm.kv_full[iv % C::STAGES], (iv / C::STAGES) & 1, sm.abort_flag)) break;
      uint4* tile = reinterpret_cast<uint4*>(sm.smem + C::OFF_KV + (iv % C::STAGES) * C::KV_BYTES);
      const int rows_valid = c.klim - j * C::BN;  // keys of this block inside the key limit
      if (rows_valid >= C::BN)
        convert_v_f16<false, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct);
      else
        convert_v_f16<true, C::KV_BYTES / 16, C::CONV_THREADS>(tile, rows_valid, ct);
      fence_proxy_async_smem();
      mbar_arrive(&sm.v_ready[iv % C::STAGES]);
    }
  } else {
    // ------------------------------------------------ softmax (warps 4-11)
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row_start = c.q0 + t * C::BM;
    const int r = row_start + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = c.tmem + lane_off + t * 128;
    const uint32_t tO = c.tmem + lane_off + 256 + t * D;
    float m_used, l;
    bool ok = fwd_softmax_pass<D, CAUSAL, false>(sm, c, t, r, tS, tO, args.s.scale_log2, 0, m_used, l);
    if (c.n_t[t] > 0 && ok) {
      ok = mbar_wait(&sm.o_full[t], 0, sm.abort_flag);
      tc_fence_after();
    }
    if (((c.own >> t) & 1) && row_start < c.sv.Lq) {
      const float omax = fwd_epilogue<D, VARLEN>(args, c, r, tO, c.n_t[t] > 0, m_used, l, 1.f);
      // Range check: a row that needs the bf16 pass flags its tile (what was
      // written is then overwritten).
      if (ok && r < c.sv.Lq && row_needs_bf16_pass(omax, l)) atomicOr(const_cast<uint32_t*>(sm.redo), 1u << t);
    }
  }

  tc_fence_before();
  __syncthreads();  // also the point where every thread learns the flagged tiles
  const uint32_t mask = *sm.redo;
  if (mask != 0) {
    tc_fence_after();
    fwd_bf16_pass<D, CAUSAL, VARLEN>(&tmK, &tmV, args, c, mask);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, C::TMEM_COLS);
  }
}

cudaError_t set_fwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_fwd_status() { return take_status_here(); }

// L2 size of the current device in bytes (0 if unknown), read once per device.
static long long current_l2_bytes() {
  constexpr int kMaxDevices = 64;
  static std::atomic<long long> cached[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  long long v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int x = 0;
    if (cudaDeviceGetAttribute(&x, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
    v = x;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// SM count of the current device, read once per device.
static long long current_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<long long> cached[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  long long v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int x = 0;
    if (cudaDeviceGetAttribute(&x, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    v = x;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

template <int D, bool CAUSAL, bool VARLEN>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdArgs& args, cudaStream_t stream, const LaunchMarks* marks) {
  using C = FwdCfg<D>;
  FwdArgs a = args;
  auto kern = fa_fwd_kernel<D, CAUSAL, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int BH = a.s.B * a.s.H;
  // Heads per group: at most as many as keep their K and V (bf16, 4 d bytes
  // per key row; the longest sequence for a packed batch) within half the L2,
  // the rest of it left to the Q tiles and the outputs streaming through;
  // groups of equal size.
  {
    const long long per_head = static_cast<long long>(std::max(a.s.Nk, 1)) * D * 4;
    const long long l2 = current_l2_bytes();
    const long long g = l2 > 0 ? (l2 / 2) / per_head : BH;
    a.heads_per_group = balanced_heads_per_group(BH, g);
  }
  const int n_pairs = (a.s.N + 2 * C::BM - 1) / (2 * C::BM);
  const long long pairs = static_cast<long long>(n_pairs) * BH;
  // Without a causal mask every pair is the same work: when the pairs leave
  // a last, partly filled wave of CTAs whose tiles fit one wave as
  // single-tile CTAs, those pairs are split, and the last wave takes about
  // half as long. (Causal grids end with their lightest pairs already.)
  long long blocks = pairs;
  if (!CAUSAL) {
    const long long sms = current_sm_count();
    const long long rem = sms > 0 ? pairs % sms : 0;
    if (rem > 0 && 2 * rem <= sms) blocks = pairs + rem;
  }
  if (blocks > 0x7fffffffLL || 2 * pairs - blocks < 0) return cudaErrorInvalidConfiguration;
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
