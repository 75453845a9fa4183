// FP8 (E4M3) forward with per-block scales, and the block quantiser feeding it.
//
// "flash_attention.zh" §9.2 (youngju.dev): FP8 tensor cores with block
// quantisation, each block keeping its own scale factor; "FlashAttention 完整
// 解析" §5.5: E4M3 inputs (range +-448), scaling before the softmax products
// so that small values do not underflow.
//
// Quantiser: per (batch, head, 128-row block) s = amax / 448 and codes
// e4m3(x * (448 / amax)) (fp32 products, round to nearest even, saturating).
// V is written transposed ([B, H, d, Np], keys contiguous) so that the P.V
// product reads both operands K-major.
//
// Forward (one CTA = two 128-row Q tiles of one (b, h), d = 128), the schedule
// of the bf16 forward with 8-bit operands:
//   S_t = Q8_t K8_j^T      tcgen05 kind::f8f6f4, fp32 in TMEM; the logits are
//                          S * scale * sQ_t * sK_j.
//   P'  = e4m3(p * 2^7 * sV_j / max_b sV_b)   with p = 2^(x - m) against the
//                          running maximum m, which is raised only when a
//                          block's maximum exceeds it by more than one binade
//                          (so p <= 2 and P' <= 256 < 448: no saturation).
//                          Folding sV_j into P' lets the accumulator run over
//                          all key blocks with one final factor.
//   O_t += P'_t V8T_j     A = P' from TMEM (32 columns), B = V^T tile K-major.
//   O = O_acc * (max sV / 2^7) / l,  l = sum of the unrounded p,  LSE = m + log l.
// Warps: 0 TMA, 1 MMA issuer, 2 the head's largest V scale, 4-11 softmax.
#include "common.cuh"
#include "ptx.cuh"

namespace fa {

// ---------------------------------------------------------------------------
// Block quantiser. One CTA per (128-row block, b*h); thread = part of a row.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_quantize_fp8_kernel(const QuantArgs a) {
  constexpr int PER = 128 * D / 256;  // values per thread
  constexpr int TPR = D / PER;        // threads per row
  __shared__ float red[8];
  __shared__ __align__(16) uint8_t tile[D * 128];  // transposed codes [D][128]
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int nb = gridDim.x;
  const int tid = threadIdx.x;
  const int r = tid / TPR;
  const int c0 = (tid % TPR) * PER;
  const int row = blk * 128 + r;
  const bool real = row < a.N;
  float v[PER];
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                    (static_cast<size_t>(bh) * a.N + (real ? row : 0)) * D + c0);
#pragma unroll
  for (int i = 0; i < PER / 8; ++i) {
    const uint4 w = real ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(ww[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  if (tid == 0) a.scale[static_cast<size_t>(bh) * nb + blk] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  uint32_t codes[PER / 4];
#pragma unroll
  for (int k = 0; k < PER / 4; ++k)
    codes[k] = pack_e4m3x4(__fmul_rn(v[4 * k], inv), __fmul_rn(v[4 * k + 1], inv), __fmul_rn(v[4 * k + 2], inv),
                           __fmul_rn(v[4 * k + 3], inv));
  if (!a.transpose) {
    if (real) {
      uint4* dst = reinterpret_cast<uint4*>(a.out + (static_cast<size_t>(bh) * a.N + row) * D + c0);
#pragma unroll
      for (int i = 0; i < PER / 16; ++i)
        dst[i] = make_uint4(codes[4 * i], codes[4 * i + 1], codes[4 * i + 2], codes[4 * i + 3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < PER; ++k) tile[(c0 + k) * 128 + r] = static_cast<uint8_t>(codes[k >> 2] >> (8 * (k & 3)));
    __syncthreads();
    const uint4* t16 = reinterpret_cast<const uint4*>(tile);
    for (int i = tid; i < D * 8; i += 256) {
      const int dcol = i >> 3, part = i & 7;
      reinterpret_cast<uint4*>(a.out + (static_cast<size_t>(bh) * D + dcol) * a.Np + blk * 128)[part] = t16[i];
    }
  }
}

cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
  const int nb = (a.N + 127) / 128;
  const dim3 grid(static_cast<unsigned>(nb), static_cast<unsigned>(a.BH));
  if (a.D == 64)
    fa_quantize_fp8_kernel<64><<<grid, 256, 0, stream>>>(a);
  else
    fa_quantize_fp8_kernel<128><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Forward.
// ---------------------------------------------------------------------------
struct Fp8Cfg {
  static constexpr int D = 128;
  static constexpr int BM = 128, BN = 128;
  static constexpr int TILE = 128 * 128;  // one 8-bit [128 x 128] tile, 128B-swizzled
  static constexpr int STAGES = 8;        // K / V^T ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE;
  static constexpr int NUM_BARS = 2 + 2 * STAGES + 2 + 2 + 2 + 1 + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
};

template <bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt, const Fp8FwdArgs args) {
  using C = Fp8Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;                    // [2]
  uint64_t* kv_full = bars + 2;               // [STAGES]
  uint64_t* kv_empty = kv_full + C::STAGES;   // [STAGES]
  uint64_t* s_full = kv_empty + C::STAGES;    // [2]
  uint64_t* p_full = s_full + 2;              // [2]
  uint64_t* o_full = p_full + 2;              // [2]
  uint64_t* mma_done = o_full + 2;
  uint64_t* vmax_ready = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vmax_ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile float* vmax_slot = reinterpret_cast<volatile float*>(tmem_slot + 2);

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
  const int klim = key_limit(args.kv_lens, b, N);
  const float* sQ = args.q_scale + static_cast<size_t>(bh) * args.nb;
  const float* sK = args.k_scale + static_cast<size_t>(bh) * args.nb;
  const float* sV = args.v_scale + static_cast<size_t>(bh) * args.nb;

  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rs = q0 + t * C::BM;
    int kmax = klim;
    if (CAUSAL) kmax = min(kmax, rs + C::BM);
    n_t[t] = (rs >= N || kmax <= 0) ? 0 : (kmax + C::BN - 1) / C::BN;
  }
  const int n_max = max(n_t[0], n_t[1]);

  // Ring position idx: K_(idx/2) (even) or V^T_(idx/2) (odd) into slot
  // idx % STAGES, once its previous use has been released.
  auto load_kv = [&](int idx) {
    const int slot = idx % C::STAGES;
    const int use = idx / C::STAGES;
    if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) return false;
    mbar_arrive_expect_tx(&kv_full[slot], C::TILE);
    uint8_t* dst = smem + C::OFF_KV + slot * C::TILE;
    const int key0 = (idx >> 1) * C::BN;
    if (idx & 1)
      tma_load_3d(dst, &tmVt, &kv_full[slot], key0, 0, bh);  // V^T: 128 d-rows x 128 keys
    else
      tma_load_3d(dst, &tmK, &kv_full[slot], 0, key0, bh);   // K: 128 keys x 128 d
    return true;
  };
  auto load_q = [&](int t) {
    if (n_t[t] > 0) {
      mbar_arrive_expect_tx(&q_full[t], C::TILE);
      tma_load_3d(smem + C::OFF_Q + t * C::TILE, &tmQ, &q_full[t], 0, q0 + t * C::BM, bh);
    }
  };
  // Thread 0 (the TMA thread) initialises the barriers of the first copies
  // and issues Q_0, K_0, Q_1 and V^T_0 before the rest of the set-up.
  const int early = min(2, 2 * n_max);  // ring positions issued in the set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 + C::STAGES; ++i) mbar_init(&bars[i], 1);  // q_full, kv_full
    fence_mbar_init();
    if (!g_test_drop_loads) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmVt);
      load_q(0);
      if (early > 0) load_kv(0);
      load_q(1);
      if (early > 1) load_kv(1);
    }
    for (int i = 2 + C::STAGES; i < C::NUM_BARS; ++i) mbar_init(&bars[i], 1);
    mbar_init(&p_full[0], 128);
    mbar_init(&p_full[1], 128);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0 && !g_test_drop_loads) {
      const int total = 2 * n_max;
      int issued = early;
      while (issued < total && load_kv(issued)) ++issued;
      // Do not leave with copies in flight (matters only after an abort, when
      // the consumers stopped waiting; every issued copy lands).
      for (int idx = max(0, issued - C::STAGES); idx < issued; ++idx)
        mbar_wait_drain(&kv_full[idx % C::STAGES], (idx / C::STAGES) & 1);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (n_t[t] > 0) mbar_wait_drain(&q_full[t], 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // The whole warp runs the issuing loop (warp-uniform waits), one elected
    // lane issues and commits.
    if (n_max > 0) {
      constexpr uint32_t IDESC = idesc_e4m3_f32(128, 128);  // S: N = 128 keys; O: N = d = 128
      const uint32_t sbase = smem_u32(smem);
      // Operand descriptors (all K-major) are built once; a Q tile, a ring slot
      // or a k-step only advances the start address (sdesc_advance).
      const uint64_t dq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dkv0 = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);
      auto slot_desc = [&](int idx) { return sdesc_advance(dkv0, (idx % C::STAGES) * C::TILE); };
      auto full_wait = [&](int idx) {
        return __all_sync(0xffffffffu, mbar_wait(&kv_full[idx % C::STAGES], (idx / C::STAGES) & 1, abort_flag));
      };
      // S_t = Q_t K^T: four K = 32 steps along the 128-byte rows.
      auto issue_qk = [&](int t, int idx) {
        const uint64_t dq = sdesc_advance(dq0, t * C::TILE), dk = slot_desc(idx);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          tc_mma_ss_f8_w(tmem + t * 128, sdesc_advance(dq, kk * 32), sdesc_advance(dk, kk * 32), IDESC,
                         kk > 0 ? 1u : 0u);
      };
      // O_t (+)= P'_t V: P' from TMEM (8 columns per 32 keys), V^T K-major.
      auto issue_pv = [&](int t, int idx, bool acc) {
        const uint64_t dv = slot_desc(idx);
#pragma unroll
        for (int kk = 0; kk < C::BN / 32; ++kk)
          tc_mma_ts_f8_w(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_advance(dv, kk * 32), IDESC,
                         (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = full_wait(0);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0 && ok) {
            // Q_t is waited for just before its first product: S_0 starts
            // before Q_1 has landed.
            ok = __all_sync(0xffffffffu, mbar_wait(&q_full[t], 0, abort_flag));
            tc_fence_after();
            if (!ok) break;
            issue_qk(t, 0);
            tc_commit_w(&s_full[t]);
          }
        tc_commit_w(&kv_empty[0]);
        for (int j = 0; j < n_max && ok; ++j) {
          const int iv = 2 * j + 1, ik = 2 * j + 2;
          ok = full_wait(iv);
          tc_fence_after();
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j < n_t[t]) {
              ok = ok && __all_sync(0xffffffffu, mbar_wait(&p_full[t], j & 1, abort_flag));
              tc_fence_after();
              issue_pv(t, iv, j > 0);
              if (j == n_t[t] - 1) tc_commit_w(&o_full[t]);
            }
            if (j + 1 < n_t[t]) {
              if (!k_ready) {
                ok = ok && full_wait(ik);
                tc_fence_after();
                k_ready = true;
              }
              issue_qk(t, ik);
              tc_commit_w(&s_full[t]);
            }
          }
          if (j + 1 < n_max) tc_commit_w(&kv_empty[ik % C::STAGES]);
          tc_commit_w(&kv_empty[iv % C::STAGES]);
        }
      }
      // TMEM is freed at the end: make sure no MMA is still running then.
      tc_commit_w(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------- the head's largest V block scale
    float m = 0.f;
    for (int i = lane; i < args.nb; i += 32) m = fmaxf(m, sV[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) {
      *vmax_slot = m;
      mbar_arrive(vmax_ready);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row_start = q0 + t * C::BM;
    const int r = row_start + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const int nt = n_t[t];
    const float sq = nt > 0 ? sQ[row_start / C::BM] : 0.f;
    float vmax = 0.f;
    bool ok = true;
    if (nt > 0) {
      ok = mbar_wait(vmax_ready, 0, abort_flag);
      vmax = *vmax_slot;
    }
    float m_used = -INFINITY;  // reference max, base-2 units of the logits
    float l = 0.f;
    for (int j = 0; j < nt && ok; ++j) {
      const float sk = sK[j], sv = sV[j];
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, abort_flag));  // warp-collective TMEM ops follow
      if (!ok) break;
      tc_fence_after();
      // Logit multiplier of this block (kept positive so masked -inf stays -inf).
      const float cj = fmaxf(sh.scale_log2 * sq * sk, 1e-30f);
      // P' = p * fj with fj = 2^7 * sV_j / max sV, folded into the exponent:
      // P' = 2^(x - m + log2 fj), and l gains sum(P') / fj. A block or head of
      // zero V takes fj = 2^7 (its P' multiplies zeros).
      const float fj = (vmax > 0.f && sv > 0.f) ? 128.f * (sv / vmax) : 128.f;
      const int kb = j * C::BN;
      const bool need_mask = (kb + C::BN > klim) || (CAUSAL && kb + C::BN - 1 > row_start);
      uint32_t s[128];
      float mx;
      if (!need_mask) {
        // No masked key: the TMEM loads also reduce the row (tcgen05.ld.red).
        float m0, m1;
        tmem_ld64_max(tS + 0, *reinterpret_cast<uint32_t(*)[64]>(&s[0]), m0);
        tmem_ld64_max(tS + 64, *reinterpret_cast<uint32_t(*)[64]>(&s[64]), m1);
        tmem_wait_ld();
        mx = fmaxf(m0, m1);
      } else {
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
        const int cmax = CAUSAL ? min(klim, r + 1) : klim;  // visible keys: c < cmax
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kb + c >= cmax) s[c] = __float_as_uint(-INFINITY);
        // Row maximum: three-input max in four independent chains over
        // s[0..3] (starts), s[4..123] (15 steps of 8) and s[124..127] (tail).
        float mxa[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) mxa[a] = __uint_as_float(s[a]);
#pragma unroll
        for (int c = 4; c < 124; c += 8)
#pragma unroll
          for (int a = 0; a < 4; ++a)
            mxa[a] = max3f(mxa[a], __uint_as_float(s[c + 2 * a]), __uint_as_float(s[c + 2 * a + 1]));
        mxa[0] = max3f(mxa[0], __uint_as_float(s[124]), __uint_as_float(s[125]));
        mxa[1] = max3f(mxa[1], __uint_as_float(s[126]), __uint_as_float(s[127]));
        mx = max3f(mxa[0], mxa[1], fmaxf(mxa[2], mxa[3]));
      }
      const float m_new = fmaxf(m_used, mx * cj);
      // Lazy rescale: the reference max moves only when a logit exceeds it by
      // more than 1.75 (base 2), so P' stays below 2^(7 + 1.75) ~ 431, inside
      // E4M3's range (448). (A threshold of 1 was 0.5-1.8 % slower.)
      const bool resc = m_new > m_used + 1.75f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2(m_used - m_new);  // 0 on the first block (m_used = -inf)
        m_used = m_new;
      }
      l *= alpha;
      const float msub = ((m_used == -INFINITY) ? 0.f : m_used) - log2f(fj);
      // x = S * cj - msub two at a time (packed fp32), then P' = 2^x.
      const uint64_t c2 = f2_pack(cj, cj), nm2 = f2_pack(-msub, -msub);
      uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // row sum of P', four independent packed chains
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), c2, nm2), x0, x1);
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), c2, nm2), x2, x3);
        const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
        rs2[i & 3] = f2_add(rs2[i & 3], f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
        pk[i] = pack_e4m3x4(p0, p1, p2, p3);
      }
      float ra, rb;
      f2_unpack(f2_add(f2_add(rs2[0], rs2[1]), f2_add(rs2[2], rs2[3])), ra, rb);
      const float blk_sum = (ra + rb) / fj;  // this block's sum of p
      tmem_st32(tS, pk);
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
      l += blk_sum;
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    // ----------------------------------------------------------- epilogue
    if (nt > 0 && ok) {
      ok = mbar_wait(&o_full[t], 0, abort_flag);
      tc_fence_after();
    }
    if (row_start < N) {
      const bool valid = r < N;
      const float inv = (l > 0.f) ? (vmax * (1.f / 128.f)) / l : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) +
                                             (static_cast<size_t>(bh) * N + r) * D);
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
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            orow[c * 4 + v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
      }
      if (valid) args.lse[static_cast<size_t>(bh) * N + r] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool CAUSAL>
static cudaError_t launch_fwd_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                                    const Fp8FwdArgs& a, cudaStream_t stream, const LaunchMarks* marks) {
  using C = Fp8Cfg;
  auto kern = fa_fwd_fp8_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int BH = a.s.B * a.s.H;
  const int n_pairs = (a.s.N + 2 * C::BM - 1) / (2 * C::BM);
  const long long blocks = static_cast<long long>(n_pairs) * BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  mark(marks, true, 0, stream);
  kern<<<static_cast<unsigned>(blocks), C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tvt, a);
  mark(marks, false, 0, stream);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8FwdArgs& a,
                           cudaStream_t stream, const LaunchMarks* m) {
  return a.s.causal ? launch_fwd_fp8_t<true>(tq, tk, tvt, a, stream, m)
                    : launch_fwd_fp8_t<false>(tq, tk, tvt, a, stream, m);
}

cudaError_t set_fp8_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream) {
  return set_test_hooks_here(wait_limit_ns, drop_loads, stream);
}

int take_fp8_status() { return take_status_here(); }

}  // namespace fa
