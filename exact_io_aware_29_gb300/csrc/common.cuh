// Shared host/device definitions of the attention library (kernel-side view).
#pragma once
#include <algorithm>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Problem description handed to every kernel (by value).
struct AttnShape {
  int B, H, N, D;    // N: (longest) query sequence length
  int Nk;            // (longest) key sequence length; = N for the fixed layout
  int causal;
  float scale;       // softmax scale applied to Q K^T
  float scale_log2;  // scale * log2(e): logits in base-2 units
};

// Where the (sequence, head) problems live. Fixed layout: [B,H,N,d], every
// sequence N long (keys optionally cut at kv_lens[b]), causal top-left.
// Packed layout (varlen = 1): [total, H, d] with sequence b at rows
// cu_q[b]..cu_q[b+1] (queries) and cu_k[b]..cu_k[b+1] (keys), N = the longest
// query sequence, causal bottom-right (query i sees key c iff c <= i + Lk - Lq).
struct Packing {
  int varlen;
  const int* cu_q;  // device int32 [B+1]
  const int* cu_k;  // device int32 [B+1]
  int total_q, total_k;
};

// One CTA's sequence: offsets and lengths, and the causal shift Lk - Lq.
struct SeqView {
  int q_start, k_start, Lq, Lk, shift;
};

// The kernels are compiled once per layout (VARLEN), so the fixed layout
// carries no packed-layout arithmetic.
template <bool VARLEN>
__device__ __forceinline__ SeqView seq_view(const Packing& pk, const int* kv_lens, int b, int N) {
  SeqView v;
  if constexpr (VARLEN) {
    v.q_start = pk.cu_q[b];
    v.Lq = pk.cu_q[b + 1] - v.q_start;
    v.k_start = pk.cu_k[b];
    v.Lk = pk.cu_k[b + 1] - v.k_start;
    v.shift = v.Lk - v.Lq;
  } else {
    int L = kv_lens == nullptr ? N : kv_lens[b];
    v.q_start = 0;
    v.k_start = 0;
    v.Lq = N;
    v.Lk = L < 0 ? 0 : (L > N ? N : L);
    v.shift = 0;
  }
  return v;
}

// Row index (in units of D elements) of row n of sequence view v, head h
// (flattened head bh = b * H + h) in a user tensor, and of its LSE entry.
template <bool VARLEN>
__device__ __forceinline__ size_t q_row(const Packing& pk, const AttnShape& s, const SeqView& v, int bh, int n) {
  return VARLEN ? (static_cast<size_t>(v.q_start) + n) * s.H + (bh % s.H) : static_cast<size_t>(bh) * s.N + n;
}
template <bool VARLEN>
__device__ __forceinline__ size_t k_row(const Packing& pk, const AttnShape& s, const SeqView& v, int bh, int n) {
  return VARLEN ? (static_cast<size_t>(v.k_start) + n) * s.H + (bh % s.H) : static_cast<size_t>(bh) * s.N + n;
}
template <bool VARLEN>
__device__ __forceinline__ size_t lse_index(const Packing& pk, const AttnShape& s, const SeqView& v, int bh, int n) {
  return VARLEN ? static_cast<size_t>(bh % s.H) * pk.total_q + v.q_start + n : static_cast<size_t>(bh) * s.N + n;
}

struct FwdArgs {
  AttnShape s;
  Packing pk;
  const int* kv_lens;    // device [B] or nullptr (fixed layout only)
  void* o;               // bf16 [B,H,N,D]
  float* lse;            // fp32 [B,H,N], natural log
  int heads_per_group;   // set at launch: heads whose CTAs run together (their K/V fit the L2)
};

struct BwdArgs {
  AttnShape s;
  Packing pk;
  const int* kv_lens;
  const void* q;       // bf16 [B,H,N,D] (plain loads for the tail paths)
  const void* o;       // bf16 [B,H,N,D]
  const float* lse;    // fp32 [B,H,N]
  const void* dO;      // bf16 [B,H,N,D]
  void* dq;            // bf16 [B,H,N,D]
  void* dk;            // bf16 [B,H,N,D]
  void* dv;            // bf16 [B,H,N,D]
  float* delta;        // workspace fp32 [B,H,N]: rowsum(dO * O)
  float* lse2;         // workspace fp32 [B,H,Np]: -LSE * log2(e) (-inf for empty and padding rows)
  float* dq_acc;       // workspace fp32 [B,H,N,D]
  // Deterministic order only (zeroed by the pre-pass in every mode):
  uint32_t* dq_turn;   // workspace u32 [B*H, Np/128]: key blocks added so far to each dQ tile
  uint32_t* ticket;    // workspace u32: next work item to hand to a starting CTA
  int deterministic;   // 1: dQ tiles summed in a fixed (descending) key-block order
  int heads_per_group; // set at launch: heads whose work items run together (L2-sized)
};

// FP8 (E4M3) block quantisation of one bf16 tensor (fp8.cu).
struct QuantArgs {
  const void* x;      // bf16 [BH, N, D]
  uint8_t* out;       // e4m3 [BH, N, D], or [BH, D, Np] when transposed
  float* scale;       // fp32 [BH, nb]: amax / 448 per 128-row block
  int BH, N, D, Np;   // Np: N rounded up to 128 (row length of the transposed form)
  int transpose;
};

// FP8 forward (fp8.cu): E4M3 Q, K [B,H,N,D] and V^T [B,H,D,Np], one fp32
// dequantisation scale per 128-row block of each.
struct Fp8FwdArgs {
  AttnShape s;
  const int* kv_lens;   // device [B] or nullptr
  const float* q_scale;  // [B*H, nb]
  const float* k_scale;
  const float* v_scale;
  int nb;               // 128-row blocks per head
  void* o;              // bf16 [B,H,N,D]
  float* lse;           // fp32 [B,H,N], natural log
};

// One decoding step over a paged KV cache (decode.cu).
struct DecodeArgs {
  const void* q;            // bf16 [B, H, D]
  void* o;                  // bf16 [B, H, D]
  float* lse;               // fp32 [B, H], natural log
  const int* block_table;   // int32 [B, max_blocks]
  const int* seq_lens;      // int32 [B], clamped to [0, max_seq_len]
  int B, H, D;
  int block_size, num_blocks, max_blocks, max_seq_len;
  int chunk, nsplit;        // keys per CTA (multiple of 64) and CTAs per (b, h)
  float scale_log2;         // scale * log2(e)
  float* part_o;            // workspace fp32 [B*H, nsplit, D] (nsplit > 1)
  float* part_ml;           // workspace fp32 [B*H, nsplit, 2]: running max (base 2), sum
};

// Key limit of batch b: keys c >= limit are masked (clamped to [0, N]).
__device__ __forceinline__ int key_limit(const int* kv_lens, int b, int N) {
  if (kv_lens == nullptr) return N;
  int L = kv_lens[b];
  return L < 0 ? 0 : (L > N ? N : L);
}

// Optional CUDA events recorded around each kernel a launcher issues
// (index = kernel order within the call); nullptr = no timing.
struct LaunchMarks {
  cudaEvent_t start[3];
  cudaEvent_t stop[3];
};

inline void mark(const LaunchMarks* m, bool start, int i, cudaStream_t s) {
  if (m != nullptr) cudaEventRecord(start ? m->start[i] : m->stop[i], s);
}

// Heads per group for a grid that runs its heads in groups (each group's
// work heaviest first, groups one after another): at most ``g_max`` heads,
// split into groups of equal size. A last group much smaller than the others
// would start its heaviest tiles only when the rest of the grid is nearly
// done and leave most SMs idle meanwhile.
inline int balanced_heads_per_group(long long bh, long long g_max) {
  if (bh <= 0) return 1;
  g_max = std::min(std::max(g_max, 1LL), bh);
  const long long groups = (bh + g_max - 1) / g_max;
  return static_cast<int>((bh + groups - 1) / groups);
}

// Launch ``kern`` on ``stream``, with programmatic stream serialization when
// ``pdl`` (the kernel may then start before the previous kernel on the stream
// has finished, and must call griddepcontrol.wait before reading its
// results). Returns the launch's error.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_maybe_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Host launchers (defined in fwd.cu / bwd.cu). Return cudaError_t of the launch.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                       cudaStream_t stream, const LaunchMarks* marks);
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream, const LaunchMarks* marks);
// Fixed device scratch of the allocation-free backward (defined in bwd.cu):
// its device address for the current device (looked up once per device) and
// its size in bytes.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
cudaError_t noalloc_scratch(void** ptr, size_t* bytes);

// Set the test hooks (wait bound, dropped loads) of each kernel translation
// unit, ordered on ``stream``.
cudaError_t set_fwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream);
cudaError_t set_bwd_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream);

// Read and clear the device status word of each kernel translation unit.
int take_fwd_status();
int take_bwd_status();
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t stream,
                          const LaunchMarks* marks);
cudaError_t set_decode_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream);
int take_decode_status();
cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8FwdArgs& a,
                           cudaStream_t stream, const LaunchMarks* marks);
cudaError_t set_fp8_test_hooks(unsigned long long wait_limit_ns, int drop_loads, cudaStream_t stream);
int take_fp8_status();

}  // namespace fa
