// C ABI of the attention library: argument checks, TMA tensor-map encoding and
// kernel launches on the caller's stream. No device memory is allocated here.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "fa_gb300.h"

namespace {

thread_local char g_last_cuda_error[256] = "no error";

int launch_error(cudaError_t e) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return FA_ERR_LAUNCH;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor maps are cached per (address, type, extents, strides, box, swizzle):
// a call with the same buffers reuses the encoded map. The cache is shared by
// all threads (behind a mutex) and emptied when it reaches kMapCacheSize.
struct MapKey {
  uintptr_t ptr;
  int dtype, swizzle;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dtype == o.dtype && swizzle == o.swizzle &&
           std::memcmp(dims, o.dims, sizeof(dims)) == 0 && std::memcmp(strides, o.strides, sizeof(strides)) == 0 &&
           std::memcmp(box, o.box, sizeof(box)) == 0;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    auto mix = [&h](uint64_t v) { h = (h ^ v) * 0x100000001B3ull; };
    mix(static_cast<uint64_t>(k.dtype));
    mix(static_cast<uint64_t>(k.swizzle));
    for (uint64_t d : k.dims) mix(d);
    for (uint64_t st : k.strides) mix(st);
    for (uint32_t b : k.box) mix(b);
    return static_cast<size_t>(h);
  }
};
constexpr size_t kMapCacheSize = 512;

bool encode_3d(CUtensorMap* m, CUtensorMapDataType dtype, const void* ptr, const uint64_t dims[3],
               const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
  MapKey key{reinterpret_cast<uintptr_t>(ptr), static_cast<int>(dtype), static_cast<int>(swizzle), {}, {}, {}};
  for (int i = 0; i < 3; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  key.strides[0] = strides[0];
  key.strides[1] = strides[1];
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *m = it->second;
      return true;
    }
  }
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  // The encoder is a driver call: a host thread that has made no CUDA runtime
  // call yet has no current context, and the encode then fails. Binding the
  // current device's primary context first (cudaSetDevice does since CUDA 12)
  // makes the library callable from any host thread.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, dtype, 3, const_cast<void*>(ptr), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() >= kMapCacheSize) cache.clear();
  cache.emplace(key, *m);
  return true;
}

// 3-D map over a [BH, N, D] bf16 tensor: box = 64 columns (128 B, the swizzle
// width) x box_rows rows x 1 slice (rows past N read as zero).
bool encode_bhnd(CUtensorMap* m, const void* ptr, int BH, int N, int D, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(N) * D * 2};
  const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a packed [total, H, D] bf16 tensor: box = 64 columns x 1 head x
// box_rows tokens (rows past `total` read as zero).
bool encode_thd(CUtensorMap* m, const void* ptr, int H, int total, int D, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H), static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(H) * D * 2};
  const uint32_t box[3] = {64, 1, static_cast<uint32_t>(box_rows)};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over an 8-bit tensor [dim2][dim1][dim0] (dim0 contiguous, row
// pitch stride1 bytes, slice pitch stride2 bytes); box = 128 x 128 x 1 with a
// 128-byte swizzle (one 128-byte row per box row).
bool encode_u8(CUtensorMap* m, const void* ptr, long long dim0, long long dim1, long long dim2, long long stride1,
               long long stride2) {
  const uint64_t dims[3] = {static_cast<uint64_t>(dim0), static_cast<uint64_t>(dim1), static_cast<uint64_t>(dim2)};
  const uint64_t strides[2] = {static_cast<uint64_t>(stride1), static_cast<uint64_t>(stride2)};
  const uint32_t box[3] = {128, 128, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Check mode: copy cu_seqlens to the host and validate them.
int check_cu_seqlens(const int* cu, int batch, int total, int max_len, cudaStream_t stream);

bool check_mode() {
  static int mode = -1;
  if (mode < 0) {
    const char* e = std::getenv("FA_CHECK");
    mode = (e != nullptr && e[0] != '\0' && e[0] != '0') ? 1 : 0;
  }
  return mode == 1;
}

int check_shape(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems > (1LL << 40) || static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Check mode: copy kv_lens to the host and validate them.
int check_kv_lens(const int* kv_lens, int B, int N, cudaStream_t stream) {
  if (kv_lens == nullptr || !check_mode()) return FA_OK;
  std::vector<int> h(B);
  cudaError_t e = cudaMemcpyAsync(h.data(), kv_lens, sizeof(int) * B, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return launch_error(e);
  for (int b = 0; b < B; ++b)
    if (h[b] < 0 || h[b] > N) return FA_ERR_INVALID;
  return FA_OK;
}

int check_cu_seqlens(const int* cu, int batch, int total, int max_len, cudaStream_t stream) {
  if (!check_mode()) return FA_OK;
  std::vector<int> h(batch + 1);
  cudaError_t e = cudaMemcpyAsync(h.data(), cu, sizeof(int) * (batch + 1), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return launch_error(e);
  if (h[0] != 0 || h[batch] != total) return FA_ERR_INVALID;
  for (int b = 0; b < batch; ++b)
    if (h[b + 1] < h[b] || h[b + 1] - h[b] > max_len) return FA_ERR_INVALID;
  return FA_OK;
}

fa::AttnShape make_shape(int B, int H, int N, int d, float scale, int causal) {
  fa::AttnShape s;
  s.B = B;
  s.H = H;
  s.N = N;
  s.D = d;
  s.Nk = N;
  s.causal = causal ? 1 : 0;
  s.scale = scale;
  s.scale_log2 = scale * fa::kLog2e;
  return s;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// How a decoding step splits each sequence's keys over CTAs: about 1024 CTAs
// in all (several waves on the GPU), chunks of whole 64-key tiles. Computed
// from the shapes alone, so the workspace size does not depend on the device.
struct DecodePlan {
  int nsplit, chunk;
};
DecodePlan decode_plan(int B, int H, int max_seq_len) {
  const long long bh = static_cast<long long>(B) * H;
  const long long tiles = (static_cast<long long>(max_seq_len) + 63) / 64;
  long long ns = (1024 + bh - 1) / bh;
  if (ns > tiles) ns = tiles;
  if (ns < 1) ns = 1;
  long long chunk = ((max_seq_len + ns - 1) / ns + 63) / 64 * 64;
  if (chunk < 64) chunk = 64;
  const long long n = (max_seq_len + chunk - 1) / chunk;
  return DecodePlan{static_cast<int>(n < 1 ? 1 : n), static_cast<int>(chunk)};
}

// Check mode: copy seq_lens and the block table to the host and validate them.
int check_decode_tables(const int* seq_lens, const int* table, int B, int max_blocks, int block_size,
                        int num_blocks, int max_seq_len, cudaStream_t stream) {
  if (!check_mode()) return FA_OK;
  std::vector<int> lens(B), tab(static_cast<size_t>(B) * max_blocks);
  cudaError_t e = cudaMemcpyAsync(lens.data(), seq_lens, sizeof(int) * B, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(tab.data(), table, sizeof(int) * tab.size(), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return launch_error(e);
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || lens[b] > max_seq_len) return FA_ERR_INVALID;
    for (int p = 0; p < (lens[b] + block_size - 1) / block_size; ++p) {
      const int x = tab[static_cast<size_t>(b) * max_blocks + p];
      if (x < 0 || x >= num_blocks) return FA_ERR_INVALID;
    }
  }
  return FA_OK;
}

// Test hooks, read from the environment on every call: FA_TEST_WAIT_LIMIT_NS
// bounds each device wait (default 2 s), FA_TEST_DROP_LOADS=1 makes the TMA
// producers issue no loads so that the dependent waits run out. Used by the
// tests of the timeout path; the device values change only when these
// variables change.
int apply_test_hooks(cudaStream_t stream) {
  static std::mutex mu;
  static unsigned long long applied_limit = 2000000000ull;
  static int applied_drop = 0;
  const char* el = std::getenv("FA_TEST_WAIT_LIMIT_NS");
  const char* ed = std::getenv("FA_TEST_DROP_LOADS");
  unsigned long long limit = 2000000000ull;
  if (el != nullptr && el[0] != '\0') {
    const unsigned long long v = std::strtoull(el, nullptr, 10);
    if (v > 0) limit = v;
  }
  const int drop = (ed != nullptr && ed[0] == '1') ? 1 : 0;
  std::lock_guard<std::mutex> lk(mu);
  if (limit == applied_limit && drop == applied_drop) return FA_OK;
  cudaError_t e = fa::set_fwd_test_hooks(limit, drop, stream);
  if (e == cudaSuccess) e = fa::set_bwd_test_hooks(limit, drop, stream);
  if (e == cudaSuccess) e = fa::set_decode_test_hooks(limit, drop, stream);
  if (e == cudaSuccess) e = fa::set_fp8_test_hooks(limit, drop, stream);
  if (e != cudaSuccess) return launch_error(e);
  applied_limit = limit;
  applied_drop = drop;
  return FA_OK;
}

// Kernel timing: pairs of CUDA events per kernel kind, filled call by call.
// 0 forward, 1 backward pre-pass, 2 backward main, 3 dQ conversion, 4 paged
// decode, 5 decode split merge, 6 FP8 forward.
constexpr int kKinds = 7;
struct Timing {
  bool on = false;
  int cap = 0;
  std::vector<cudaEvent_t> start[kKinds], stop[kKinds];
  int used[kKinds] = {0, 0, 0, 0, 0, 0, 0};
};
Timing g_timing;
std::mutex g_timing_mu;

// Event slots for the next call's kernels (first = kind of its first kernel).
bool next_marks(fa::LaunchMarks* m, int first, int count) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (!g_timing.on) return false;
  for (int i = 0; i < count; ++i)
    if (g_timing.used[first + i] >= g_timing.cap) return false;
  for (int i = 0; i < count; ++i) {
    const int k = first + i, u = g_timing.used[k]++;
    m->start[i] = g_timing.start[k][u];
    m->stop[i] = g_timing.stop[k][u];
  }
  return true;
}

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim, alignment or size";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: CUDA error";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device wait ran out";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
    case FA_ERR_SCRATCH_LIMIT:
      return "FA_ERR_SCRATCH_LIMIT: problem needs more than the fixed scratch of fa_bwd_noalloc";
    default: return "unknown fa_status";
  }
}

const char* fa_last_cuda_error(void) { return g_last_cuda_error; }

int fa_check_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return launch_error(e);
  const int a = fa::take_fwd_status();
  const int b = fa::take_bwd_status();
  const int c = fa::take_decode_status();
  const int f = fa::take_fp8_status();
  if (a == FA_ERR_LAUNCH || b == FA_ERR_LAUNCH || c == FA_ERR_LAUNCH || f == FA_ERR_LAUNCH)
    return launch_error(cudaGetLastError());
  if (a != 0 || b != 0 || c != 0 || f != 0) return FA_ERR_TIMEOUT;
  return FA_OK;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, const int* kv_lens, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID;
  int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_kv_lens(kv_lens, B, N, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!encode_bhnd(&tq, q, BH, N, d, 128) || !encode_bhnd(&tk, k, BH, N, d, 128) ||
      !encode_bhnd(&tv, v, BH, N, d, 128))
    return launch_error(cudaErrorInvalidValue);
  fa::FwdArgs a;
  a.s = make_shape(B, H, N, d, scale, causal);
  a.pk = fa::Packing{0, nullptr, nullptr, 0, 0};
  a.kv_lens = kv_lens;
  a.o = o;
  a.lse = lse;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 0, 1);
  cudaError_t e = fa::launch_fwd(tq, tk, tv, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int batch, int H, int d, int total_q, int total_k, int max_seqlen_q,
                  int max_seqlen_k, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID;
  if (total_q < 1 || total_k < 1 || max_seqlen_q < 1 || max_seqlen_k < 1) return FA_ERR_INVALID;
  if (max_seqlen_q > total_q || max_seqlen_k > total_k) return FA_ERR_INVALID;
  int st = check_shape(batch, H, max_seqlen_q, d, scale);
  if (st != FA_OK) return st;
  if (static_cast<long long>(total_q) * H * d > (1LL << 40) || static_cast<long long>(total_k) * H * d > (1LL << 40))
    return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_cu_seqlens(cu_seqlens_q, batch, total_q, max_seqlen_q, s);
  if (st == FA_OK) st = check_cu_seqlens(cu_seqlens_k, batch, total_k, max_seqlen_k, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  CUtensorMap tq, tk, tv;
  if (!encode_thd(&tq, q, H, total_q, d, 128) || !encode_thd(&tk, k, H, total_k, d, 128) ||
      !encode_thd(&tv, v, H, total_k, d, 128))
    return launch_error(cudaErrorInvalidValue);
  fa::FwdArgs a;
  a.s = make_shape(batch, H, max_seqlen_q, d, scale, causal);
  a.pk = fa::Packing{1, cu_seqlens_q, cu_seqlens_k, total_q, total_k};
  a.kv_lens = nullptr;
  a.o = o;
  a.lse = lse;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 0, 1);
  cudaError_t e = fa::launch_fwd(tq, tk, tv, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 1.f) != FA_OK) return 0;
  // Rows are padded per head to whole 128-row blocks.
  const size_t rows = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128 * 128);
  return align_up(rows * 4, 256) * 2 + align_up(rows * d * 4, 256) + align_up(rows / 128 * 4, 256) + 256;
}

// Carves the workspace: delta, -LSE*log2(e), the dQ accumulator, then the
// per-block counters and the ticket of the deterministic order.
static void carve_workspace(fa::BwdArgs* a, void* workspace, size_t rows, int d) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t vec = align_up(rows * 4, 256), acc = align_up(rows * d * 4, 256);
  a->delta = reinterpret_cast<float*>(ws);
  a->lse2 = reinterpret_cast<float*>(ws + vec);
  a->dq_acc = reinterpret_cast<float*>(ws + 2 * vec);
  a->dq_turn = reinterpret_cast<uint32_t*>(ws + 2 * vec + acc);
  a->ticket = reinterpret_cast<uint32_t*>(ws + 2 * vec + acc + align_up(rows / 128 * 4, 256));
}

static int bwd_fixed(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                     const int* kv_lens, void* workspace, size_t workspace_bytes, void* stream, int det) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID;
  int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_kv_lens(kv_lens, B, N, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_bhnd(&tq, q, BH, N, d, 128) || !encode_bhnd(&tk, k, BH, N, d, 128) ||
      !encode_bhnd(&tv, v, BH, N, d, 128) || !encode_bhnd(&tdo, dO, BH, N, d, 128))
    return launch_error(cudaErrorInvalidValue);
  const size_t rows = static_cast<size_t>(BH) * ((static_cast<size_t>(N) + 127) / 128 * 128);
  fa::BwdArgs a;
  a.s = make_shape(B, H, N, d, scale, causal);
  a.pk = fa::Packing{0, nullptr, nullptr, 0, 0};
  a.kv_lens = kv_lens;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  carve_workspace(&a, workspace, rows, d);
  a.deterministic = det;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 1, 3);
  cudaError_t e = fa::launch_bwd(tq, tk, tv, tdo, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
           const int* kv_lens, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_fixed(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, kv_lens, workspace,
                   workspace_bytes, stream, 0);
}

int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const int* kv_lens, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_fixed(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, kv_lens, workspace,
                   workspace_bytes, stream, 1);
}

int fa_timing_end(void) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  for (int k = 0; k < kKinds; ++k) {
    for (cudaEvent_t ev : g_timing.start[k]) cudaEventDestroy(ev);
    for (cudaEvent_t ev : g_timing.stop[k]) cudaEventDestroy(ev);
    g_timing.start[k].clear();
    g_timing.stop[k].clear();
    g_timing.used[k] = 0;
  }
  g_timing.on = false;
  g_timing.cap = 0;
  return FA_OK;
}

int fa_timing_begin(int max_calls) {
  if (max_calls < 1 || max_calls > (1 << 20)) return FA_ERR_INVALID;
  fa_timing_end();
  std::lock_guard<std::mutex> lk(g_timing_mu);
  for (int k = 0; k < kKinds; ++k) {
    g_timing.start[k].assign(max_calls, nullptr);
    g_timing.stop[k].assign(max_calls, nullptr);
    for (int i = 0; i < max_calls; ++i) {
      cudaError_t e = cudaEventCreate(&g_timing.start[k][i]);
      if (e == cudaSuccess) e = cudaEventCreate(&g_timing.stop[k][i]);
      if (e != cudaSuccess) return launch_error(e);
    }
  }
  g_timing.cap = max_calls;
  g_timing.on = true;
  return FA_OK;
}

int fa_timing_read(int kind, double* total_ms, int* count) {
  if (kind < 0 || kind >= kKinds || total_ms == nullptr || count == nullptr) return FA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  double tot = 0.0;
  const int n = g_timing.used[kind];
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(g_timing.stop[kind][i]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_timing.start[kind][i], g_timing.stop[kind][i]);
    if (e != cudaSuccess) return launch_error(e);
    tot += ms;
  }
  *total_ms = tot;
  *count = n;
  return FA_OK;
}

// Backward without any device allocation: the workspace is the library's
// fixed static scratch (see fa_bwd_noalloc in the header).
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                   const int* kv_lens, void* stream) {
  const int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (fa_bwd_workspace_size(B, H, N, d) > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  size_t bytes = 0;
  const cudaError_t e = fa::noalloc_scratch(&scratch, &bytes);
  if (e != cudaSuccess) return launch_error(e);
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, kv_lens, scratch, bytes, stream);
}

static int bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, int batch, int H, int d, int total_q, int total_k, int max_seqlen_q,
                      int max_seqlen_k, float scale, int causal, void* workspace, size_t workspace_bytes,
                      void* stream, int det) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_k)
    return FA_ERR_INVALID;
  if (total_q < 1 || total_k < 1 || max_seqlen_q < 1 || max_seqlen_k < 1) return FA_ERR_INVALID;
  if (max_seqlen_q > total_q || max_seqlen_k > total_k) return FA_ERR_INVALID;
  int st = check_shape(batch, H, max_seqlen_q, d, scale);
  if (st != FA_OK) return st;
  if (static_cast<long long>(total_q) * H * d > (1LL << 40) || static_cast<long long>(total_k) * H * d > (1LL << 40))
    return FA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_bwd_workspace_size(batch, H, max_seqlen_q, d);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_cu_seqlens(cu_seqlens_q, batch, total_q, max_seqlen_q, s);
  if (st == FA_OK) st = check_cu_seqlens(cu_seqlens_k, batch, total_k, max_seqlen_k, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_thd(&tq, q, H, total_q, d, 128) || !encode_thd(&tk, k, H, total_k, d, 128) ||
      !encode_thd(&tv, v, H, total_k, d, 128) || !encode_thd(&tdo, dO, H, total_q, d, 128))
    return launch_error(cudaErrorInvalidValue);
  const size_t rows = static_cast<size_t>(batch) * H * ((static_cast<size_t>(max_seqlen_q) + 127) / 128 * 128);
  fa::BwdArgs a;
  a.s = make_shape(batch, H, max_seqlen_q, d, scale, causal);
  a.s.Nk = max_seqlen_k;
  a.pk = fa::Packing{1, cu_seqlens_q, cu_seqlens_k, total_q, total_k};
  a.kv_lens = nullptr;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  carve_workspace(&a, workspace, rows, d);
  a.deterministic = det;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 1, 3);
  cudaError_t e = fa::launch_bwd(tq, tk, tv, tdo, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int H,
                  int d, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, float scale, int causal,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, H, d, total_q, total_k,
                    max_seqlen_q, max_seqlen_k, scale, causal, workspace, workspace_bytes, stream, 0);
}

int fa_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                                const int* cu_seqlens_k, int batch, int H, int d, int total_q, int total_k,
                                int max_seqlen_q, int max_seqlen_k, float scale, int causal, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, H, d, total_q, total_k,
                    max_seqlen_q, max_seqlen_k, scale, causal, workspace, workspace_bytes, stream, 1);
}

size_t fa_decode_workspace_size(int B, int H, int d, int max_seq_len) {
  if (check_shape(B, H, max_seq_len, d, 1.f) != FA_OK) return 0;
  const DecodePlan pl = decode_plan(B, H, max_seq_len);
  const size_t parts = static_cast<size_t>(B) * H * pl.nsplit;
  return align_up(parts * d * 4, 256) + align_up(parts * 2 * 4, 256);
}

int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const int* block_table, const int* seq_lens, int B, int H, int d, int num_blocks,
                    int block_size, int max_blocks_per_seq, int max_seq_len, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !o || !lse || !block_table || !seq_lens) return FA_ERR_INVALID;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || block_size < 1) return FA_ERR_INVALID;
  int st = check_shape(B, H, max_seq_len, d, scale);
  if (st != FA_OK) return st;
  if (block_size % 64 != 0) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_seq_len) > static_cast<long long>(max_blocks_per_seq) * block_size)
    return FA_ERR_INVALID;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_cache, v_cache, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return FA_ERR_UNSUPPORTED;
  const DecodePlan pl = decode_plan(B, H, max_seq_len);
  const size_t need = fa_decode_workspace_size(B, H, d, max_seq_len);
  if (pl.nsplit > 1 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_decode_tables(seq_lens, block_table, B, max_blocks_per_seq, block_size, num_blocks, max_seq_len, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  CUtensorMap tk, tv;
  const int rows = num_blocks * block_size;
  if (!encode_thd(&tk, k_cache, H, rows, d, 64) || !encode_thd(&tv, v_cache, H, rows, d, 64))
    return launch_error(cudaErrorInvalidValue);
  fa::DecodeArgs a;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.B = B;
  a.H = H;
  a.D = d;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.chunk = pl.chunk;
  a.nsplit = pl.nsplit;
  a.scale_log2 = scale * fa::kLog2e;
  const size_t parts = static_cast<size_t>(B) * H * pl.nsplit;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_o = pl.nsplit > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  a.part_ml = pl.nsplit > 1 ? reinterpret_cast<float*>(ws + align_up(parts * d * 4, 256)) : nullptr;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 4, pl.nsplit > 1 ? 2 : 1);
  cudaError_t e = fa::launch_decode(tk, tv, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

int fa_quantize_fp8(const void* x, void* out, float* block_scale, int B, int H, int N, int d, int transpose,
                    void* stream) {
  if (!x || !out || !block_scale) return FA_ERR_INVALID;
  int st = check_shape(B, H, N, d, 1.f);
  if (st != FA_OK) return st;
  if (!aligned16(x) || !aligned16(out)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;  // grid.y
  fa::QuantArgs a;
  a.x = x;
  a.out = static_cast<uint8_t*>(out);
  a.scale = block_scale;
  a.BH = B * H;
  a.N = N;
  a.D = d;
  a.Np = (N + 127) / 128 * 128;
  a.transpose = transpose ? 1 : 0;
  cudaError_t e = fa::launch_quantize_fp8(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
               const int* kv_lens, void* stream) {
  if (!q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale || !o || !lse) return FA_ERR_INVALID;
  int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q8, k8, v8t, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return FA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = check_kv_lens(kv_lens, B, N, s);
  if (st != FA_OK) return st;
  st = apply_test_hooks(s);
  if (st != FA_OK) return st;
  const long long BH = static_cast<long long>(B) * H;
  const long long Np = (static_cast<long long>(N) + 127) / 128 * 128;
  CUtensorMap tq, tk, tv;
  if (!encode_u8(&tq, q8, d, N, BH, d, static_cast<long long>(N) * d) ||
      !encode_u8(&tk, k8, d, N, BH, d, static_cast<long long>(N) * d) ||
      !encode_u8(&tv, v8t, Np, d, BH, Np, Np * d))
    return launch_error(cudaErrorInvalidValue);
  fa::Fp8FwdArgs a;
  a.s = make_shape(B, H, N, d, scale, causal);
  a.kv_lens = kv_lens;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.nb = static_cast<int>(Np / 128);
  a.o = o;
  a.lse = lse;
  fa::LaunchMarks marks;
  const bool timed = next_marks(&marks, 6, 1);
  cudaError_t e = fa::launch_fwd_fp8(tq, tk, tv, a, s, timed ? &marks : nullptr);
  if (e != cudaSuccess) return launch_error(e);
  if (check_mode()) return fa_check_status(stream);
  return FA_OK;
}

}  // extern "C"
