// C-ABI layer: argument validation, tensor-map encoding, path selection,
// library workspace and the device status word.  See include/gemm_tn.h.
//
// Tensor maps (Ampere-to-Hopper page, section "TMA: from copying addresses to
// copying tensor tiles": base, shape, stride, box, swizzle and out-of-bounds
// policy in one descriptor) are encoded on the host for every call: A and B
// with 64x(rows) boxes and 128-byte swizzle so that the shared-memory image
// is the canonical K-major layout the tcgen05 descriptors describe; C and D
// with 32x32 boxes for the epilogue.  Out-of-range boxes are zero-filled on
// load and clipped on store, which is how ragged M, N and K are handled.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/gemm_tn.h"
#include "kernels.h"

namespace gtn {
namespace {

// Device status word ([0] = code, [1] = detail), one copy per device.
__device__ int g_status[kStatusWords];

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// L2 hints of single-problem tiled calls without a config (kL2Hint* bits).
constexpr int kDefaultL2Hints = 0;

thread_local std::string t_error;
thread_local gemm_launch_info t_info = {};
thread_local int t_last_detail = 0;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_error = buf;
  return code;
}

struct DeviceState {
  bool ready = false;
  int cc_major = 0, cc_minor = 0, sms = 0;
  int* status = nullptr;  // device address of g_status
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

struct Workspace {
  float* partials = nullptr;
  size_t partial_floats = 0;
  int* counters = nullptr;
  size_t counter_ints = 0;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int init_device(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    st.cc_major = prop.major;
    st.cc_minor = prop.minor;
    st.sms = prop.multiProcessorCount;
    if (!(st.cc_major == 10 && st.cc_minor == 3))
      return fail(GEMM_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                  st.cc_major, st.cc_minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    st.status = static_cast<int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.ready = true;
  }
  *dev_out = dev;
  *st_out = &st;
  return GEMM_OK;
}

// 2D tensor map over a row-major matrix (inner = contiguous dimension).
int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner, uint64_t outer,
              uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw, const char* what) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld_elems * (uint64_t)esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return GEMM_OK;
}

// 3D view of a row-major matrix for loads of kg consecutive k-blocks in one
// box: dims {k in block, row, k-block}, the k-block stride being the block's
// 128 bytes.  K must be a whole number of k-blocks (the view has no zero fill
// inside a row); k-blocks past K and rows past `outer` are zero-filled.
int encode_kgroups(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t K, uint64_t outer,
                   uint64_t ld_elems, uint32_t kbe, uint32_t box_outer, uint32_t kg, const char* what) {
  cuuint64_t dims[3] = {kbe, outer, K / kbe};
  cuuint64_t strides[2] = {ld_elems * (uint64_t)esize, (uint64_t)kbe * esize};
  cuuint32_t box[3] = {kbe, box_outer, kg};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled(%s, k-groups) failed with %d", what, (int)r);
  return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t timeout_ns(const gemm_tn_config* cfg) {
  if (cfg && cfg->wait_timeout_ns) return cfg->wait_timeout_ns;
  static uint64_t env = [] {
    const char* s = getenv("GEMM_WAIT_TIMEOUT_NS");
    if (s && *s) {
      unsigned long long v = strtoull(s, nullptr, 10);
      if (v > 0) return (uint64_t)v;
    }
    return kDefaultTimeoutNs;
  }();
  return env;
}

// `optional`: the caller can do without (the tiled k-split): where the
// workspace would have to grow during stream capture, return GEMM_OK with
// *out = nullptr instead of an error.
int get_workspace(int dev, cudaStream_t stream, size_t partial_floats, size_t counter_ints, Workspace** out,
                  bool optional = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  *out = nullptr;
  Workspace& w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
  if (w.partial_floats < partial_floats || w.counter_ints < counter_ints) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cs);
    if (cs != cudaStreamCaptureStatusNone) {
      if (optional) return GEMM_OK;
      return fail(GEMM_ERR_INVALID_VALUE, "split-K workspace must be created outside stream capture");
    }
    // Work already queued may still use the old buffers.
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    if (w.partials) cudaFree(w.partials);
    if (w.counters) cudaFree(w.counters);
    w = Workspace{};
    size_t pf = partial_floats < (1u << 16) ? (1u << 16) : partial_floats;
    size_t ci = counter_ints < 4096 ? 4096 : counter_ints;
    if (cudaMalloc(&w.partials, pf * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&w.counters, ci * sizeof(int)) != cudaSuccess) {
      if (w.partials) cudaFree(w.partials);
      w = Workspace{};
      cudaGetLastError();
      return fail(GEMM_ERR_OUT_OF_MEMORY, "split-K workspace allocation failed");
    }
    e = cudaMemset(w.counters, 0, ci * sizeof(int));
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    w.partial_floats = pf;
    w.counter_ints = ci;
  }
  *out = &w;
  return GEMM_OK;
}

// Argument rules shared by every entry point for one problem's operands (the
// header states them): sizes below 2^31, D present with ldd >= N, C present
// when beta != 0, A and B present with ld >= K when K > 0, and the 16-byte
// alignment TMA needs for every base address and row pitch.
int check_operands(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   const void* C, int64_t ldc, const void* D, int64_t ldd, bool has_c, int esize, int in_bytes) {
  const int64_t kMaxDim = (int64_t)1 << 31;
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return fail(GEMM_ERR_INVALID_VALUE, "sizes must be below 2^31");
  if (!D) return fail(GEMM_ERR_INVALID_VALUE, "D is NULL");
  if (ldd < N) return fail(GEMM_ERR_INVALID_VALUE, "ldd (%lld) < N (%lld)", (long long)ldd, (long long)N);
  if (has_c) {
    if (!C) return fail(GEMM_ERR_INVALID_VALUE, "beta != 0 but C is NULL");
    if (ldc < N) return fail(GEMM_ERR_INVALID_VALUE, "ldc (%lld) < N (%lld)", (long long)ldc, (long long)N);
  }
  if (K > 0) {
    if (!A || !B) return fail(GEMM_ERR_INVALID_VALUE, "A or B is NULL");
    if (lda < K || ldb < K)
      return fail(GEMM_ERR_INVALID_VALUE, "lda (%lld) and ldb (%lld) must be >= K (%lld)", (long long)lda,
                  (long long)ldb, (long long)K);
    if (!aligned16(A) || !aligned16(B)) return fail(GEMM_ERR_MISALIGNED, "A and B must be 16-byte aligned");
    if ((lda * in_bytes) % 16 || (ldb * in_bytes) % 16)
      return fail(GEMM_ERR_MISALIGNED, "lda and ldb must be multiples of %d elements", 16 / in_bytes);
  }
  if (!aligned16(D) || (ldd * esize) % 16)
    return fail(GEMM_ERR_MISALIGNED, "D must be 16-byte aligned with ldd*%d a multiple of 16", esize);
  if (has_c && (!aligned16(C) || (ldc * esize) % 16))
    return fail(GEMM_ERR_MISALIGNED, "C must be 16-byte aligned with ldc*%d a multiple of 16", esize);
  return GEMM_OK;
}

// A GEMM of at most this many 128 x 256 tiles whose B stays in L2 runs on
// 1-SM tiles even when M > 128: with so few tiles the pair kernel's cluster
// launch costs more than its shared operand traffic saves (measured 0.5-0.8
// us per call from 256^3 to 1024 x 2048 x 2048; with 120 tiles the pair
// kernel was faster).
constexpr long long kSmallTileCount = 64;

long long one_sm_tiles(int64_t M, int64_t N) { return ((M + 127) / 128) * ((N + 255) / 256); }

// Automatic path.  The numbers are GB300 measurements (graph-replayed calls,
// B rotated over copies so that it streams from HBM where it is large), from
// `bench.py --path-check` (180 shapes against every forced choice) after the
// tiled k-split's partials were interleaved and grids under one round were
// sliced, which made the tiled kernels faster on few tiles.
// - Up to 32 tokens: the streaming kernel (swap-AB, tokens as MMA N), except
//   for short rows of a small B (K <= 1024, 1024 <= N <= 4096), where sliced
//   1-SM tiles start and finish sooner (32 x 1024 x 1024: 7.4 against 10.9
//   us; 16 x 4096 x 1024: 7.6 against 8.9).
// - 33..128 tokens: streaming where B is too large to stay in L2 between
//   calls (>= 32 MiB) and the streaming kernel splits each tile into at most
//   two k-parts.  128 x 8192 x 8192: 38.5 us against 43.6 (2-SM) and 56.6
//   (1-SM).  Where tiles fall to stream-K (64 x 28672 x 4096: 49.9 against
//   44.5 us) or B is small (64 x 4096 x 1024: 13.1 against 9.3 us), the
//   tiled kernels win.  Refinements (see auto_path): up to 64 tokens, four
//   parts with a long K also stream, but not for N <= 4096, where tiles in
//   four k-parts are faster (64 x 1024 x 4096: 17.6 against 22.6 us; 64 x
//   4096 x 8192: 27.1 against 28.9); above 64 tokens, only 4096 < N <= 8192
//   with K of at least 64 k-blocks (32 up to 96 tokens) streams (128 x 4096
//   x 8192: pair tiles in four parts 27.5 against 37.5 us; 128 x 8192 x
//   2048: 1-SM 14.6 against 16.0; 96 x 8192 x 2048: 14.7 either way).
// - When B streams from HBM and the tiles are few, pair tiles win over 1-SM
//   tiles even for M <= 128: each SM of a pair loads half of the B tile, and
//   twice the SMs stream (96 x 16384 x 8192: 53.5 against 61.6 us), unless K
//   is short (32 k-blocks or fewer: 128 x 16384 x 1024 on sliced 1-SM tiles
//   10.8 against 12.4 us).  For 129..256 tokens this holds at any tile count
//   (224 x 8192 x 8192: 44.0 against 56.6 us); with B in L2 the 1-SM
//   kernel's lighter launch wins.
constexpr int64_t kStreamedBytes = 32ll << 20;

// k-parts per tile for the tiled kernels (single problem, static schedule),
// one cluster per (tile, part); part 0 adds the other parts' fp32 partials.
// Measured on GB300 (graph-replayed, bf16, B rotated), none / two / four parts:
//   256 x 2048 x 8192 (8 pair tiles, 128 k-blocks)   40.0 / 31.7 / 24.6 us
//   256 x 4096 x 8192 (16)                            41.3 / 32.9 / 27.6
//   192 x 4096 x 4096 (16, 64 k-blocks)               22.7 / 23.2 / 21.2
//   256 x 4096 x 4096 (16, 64 k-blocks)               22.6 / 23.3 / 21.4
//   224 x 8192 x 8192 (32, 128 k-blocks)              41.8 / 38.4 / (does not fit)
//   512 x 4096 x 4096 (32, 64 k-blocks)               23.5 / 23.8 / (does not fit)
//   300 x 1096 x 4096 (15 1-SM tiles, 64 k-blocks)    24.0 / 23.9 / 19.9
//   256 x 2048 x 2048 (8, 32 k-blocks)                13.3 / 18.2 / 17.6
//   1024 x 2048 x 2048 (64 1-SM tiles, 32 k-blocks)   14.4 / 18.5 / (does not fit)
// So four parts where they fit one round of clusters and K holds at least 64
// k-blocks, else two where they fit and K holds at least 128, else none.
// Every unit needs a co-resident cluster (part 0 waits for the others).
// Forced values (tiled_k_parts) go up to four.
constexpr int kMaxTiledParts = 4;
constexpr int kFusedSplitMinKb = 128;   // fused calls: four parts of 32+ k-blocks
constexpr int kSplit4MinKb = 64;
constexpr int kSplit2MinKb = 128;
int tiled_parts(long long tiles, int num_kb, int sms, int cg, const gemm_tn_config* cfg) {
  const int req = cfg ? cfg->tiled_k_parts : 0;
  if (req > 0) return req < num_kb ? req : (num_kb > 1 ? num_kb : 1);
  const long long clusters = sms / cg;
  if (tiles < 1) return 1;
  if (4 * tiles <= clusters && num_kb >= kSplit4MinKb) return 4;
  if (2 * tiles <= clusters && num_kb >= kSplit2MinKb) return 2;
  return 1;
}

// Slices of the last round of a static tiled launch over `clusters`
// clusters: the tiles past the last whole round (all of them when they fill
// less than one round) are cut into 2^shift slices each, the most (up to 4,
// or the count cfg asks for) that still fit one round.  begin = first tile
// cut; shift = 0 when none is.  Automatic only when the tiles fill less
// than one round (small GEMMs: 256^3 6.1 -> 3.8 us, 512 x 3072 x 4096
// 32.1 -> 26.4 us).  Over several rounds the gain was small and the code
// that slices cost more than it: with slices in the kernel everything else
// ran 1-4% slower, and the launches with slices now take a kernel of their
// own.  At 8192 x 28672 x 4096 quarters of the last round's 12 tiles were
// 0.4-0.8% slower; 4096^3 and 3000 x 5000 x 2000 (3.4 and 3.2 rounds)
// gained 1.4% and 2.8% against that kernel without slices (interleaved runs).
void tail_slices_plan(long long tiles, int clusters, const gemm_tn_config* cfg, int* begin, int* shift) {
  *begin = (int)tiles;
  *shift = 0;
  const int req = cfg ? cfg->tail_slices : 0;
  if (req == 1 || tiles < 1 || clusters < 2) return;
  if (req == 0 && tiles >= clusters) return;
  const long long r = tiles % clusters;   // tiles of the last round (all of them if < clusters)
  if (r == 0) return;
  for (int sh = 2; sh >= 1; --sh) {
    if (req != 0 && req != (1 << sh)) continue;
    if ((r << sh) <= clusters) {
      *begin = (int)(tiles - r);
      *shift = sh;
      return;
    }
  }
}

// Values of a gemm_tn_config that select among fixed choices.
int check_config(const gemm_tn_config* cfg) {
  if (!cfg) return GEMM_OK;
  if (cfg->path < GEMM_PATH_AUTO || cfg->path > GEMM_PATH_SKINNY)
    return fail(GEMM_ERR_INVALID_VALUE, "unknown path %d", cfg->path);
  const int sched = cfg->scheduler;
  if (sched != GEMM_SCHED_DEFAULT && sched != GEMM_SCHED_STATIC && sched != GEMM_SCHED_CLC)
    return fail(GEMM_ERR_INVALID_VALUE, "unknown scheduler %d", sched);
  if (cfg->skinny_bm != 0 && cfg->skinny_bm != 64 && cfg->skinny_bm != 128)
    return fail(GEMM_ERR_INVALID_VALUE, "skinny_bm must be 0, 64 or 128, got %d", cfg->skinny_bm);
  const int kg = cfg->skinny_kgroup;
  if (kg != 0 && kg != 1 && kg != 2 && kg != 4)
    return fail(GEMM_ERR_INVALID_VALUE, "skinny_kgroup must be 0, 1, 2 or 4, got %d", kg);
  if (cfg->b_static != 0 && cfg->b_static != 1)
    return fail(GEMM_ERR_INVALID_VALUE, "b_static must be 0 or 1, got %d", cfg->b_static);
  if (cfg->skinny_pair < 0 || cfg->skinny_pair > 2)
    return fail(GEMM_ERR_INVALID_VALUE, "skinny_pair must be 0, 1 or 2, got %d", cfg->skinny_pair);
  if (cfg->cluster_pref != 0 && cfg->cluster_pref != 4 && cfg->cluster_pref != 8)
    return fail(GEMM_ERR_INVALID_VALUE, "cluster_pref must be 0, 4 or 8, got %d", cfg->cluster_pref);
  if (cfg->tail_slices != 0 && cfg->tail_slices != 1 && cfg->tail_slices != 2 && cfg->tail_slices != 4)
    return fail(GEMM_ERR_INVALID_VALUE, "tail_slices must be 0, 1, 2 or 4, got %d", cfg->tail_slices);
  if (cfg->l2_hints < -1 || cfg->l2_hints > 7)
    return fail(GEMM_ERR_INVALID_VALUE, "l2_hints must be -1..7, got %d", cfg->l2_hints);
  if (cfg->tiled_k_parts < 0 || cfg->tiled_k_parts > kMaxTiledParts)
    return fail(GEMM_ERR_INVALID_VALUE, "tiled_k_parts must be 0..%d, got %d", kMaxTiledParts, cfg->tiled_k_parts);
  return GEMM_OK;
}

// Automatic path for a shape on `sms` SMs (host only; rules above).
int auto_path(int64_t M, int64_t N, int64_t K, int in_bytes, int sms) {
  if (K == 0) return GEMM_PATH_1SM;
  const bool streamed = N * K * in_bytes >= kStreamedBytes;
  const int np = (int)((M + 15) / 16) * 16;
  const int parts = M <= 256 ? skinny_parts(N, np, skinny_max_grid(np, sms)) : 0;
  const long long tiles = one_sm_tiles(M, N);
  const long long num_kb = (K + 128 / in_bytes - 1) / (128 / in_bytes);
  if (M <= 32) return (num_kb <= 16 && N >= 1024 && N <= 4096) ? GEMM_PATH_1SM : GEMM_PATH_SKINNY;
  // 33..64 tokens: also on a few tiles split four ways once K is long, but
  // not where N <= 4096 (the tiled k-split in four parts is faster there)
  if (M <= 64 && parts >= 1 && ((streamed && parts <= 2 && !(N <= 4096 && num_kb >= 64)) ||
                                (num_kb >= 64 && N > 4096)))
    return GEMM_PATH_SKINNY;
  // 65..128 tokens (wide form): only for 4096 < N <= 8192 with long rows of B
  // (K of 64 k-blocks, or 32 up to 96 tokens)
  if (M > 64 && M <= 128 && streamed && parts >= 1 && parts <= 2 && N > 4096 && N <= 8192 &&
      (num_kb >= 64 || (M <= 96 && num_kb >= 32)))
    return GEMM_PATH_SKINNY;
  if (M > 128 && (streamed || tiles > kSmallTileCount)) return GEMM_PATH_2SM;
  if (M <= 128 && streamed && 2 * tiles <= sms && num_kb > 32) return GEMM_PATH_2SM;
  return GEMM_PATH_1SM;
}

// Skinny-path geometry and work partition (host only): tile rows, k-group,
// k-groups per tile, tiles, units, grid, split and skew.  Config overrides
// were validated by the caller.
int skinny_geometry(SkinnyParams* p, int64_t M, int64_t N, int64_t K, int kbe, int sms, const gemm_tn_config* cfg) {
  const int np = (int)((M + 15) / 16) * 16;
  p->M = (int)M; p->N = (int)N; p->K = (int)K; p->np = np;
  // The pair form (clusters of two CTAs, 256-row tiles, cta_group::2 MMAs,
  // half the tokens per CTA) only where asked for.
  p->cg = cfg && cfg->skinny_pair == 2 ? 2 : 1;
  const int npc = np / p->cg;  // token rows per CTA
  const int max_grid = skinny_max_grid(np, sms) / p->cg;  // CTAs, or pairs
  const int bm_req = cfg ? cfg->skinny_bm : 0, kg_req = cfg ? cfg->skinny_kgroup : 0;
  if (p->cg == 2 && bm_req && bm_req != 128)
    return fail(GEMM_ERR_INVALID_VALUE, "the pair form takes 128 rows of B per CTA (skinny_bm 0 or 128)");
  p->bm = p->cg == 2 ? 128 : (bm_req ? bm_req : skinny_tile_rows(N, np, max_grid));
  p->kg = skinny_kgroup(npc, p->bm, K, kbe, kg_req);
  if (skinny_stages(npc, p->bm, p->kg) < 2)
    return fail(GEMM_ERR_INVALID_VALUE, "skinny_kgroup %d leaves fewer than 2 ring stages at M = %lld", p->kg,
                (long long)M);
  p->stages = skinny_stages(npc, p->bm, p->kg);
  p->num_kb = (int)(((K + kbe - 1) / kbe + p->kg - 1) / p->kg);
  p->n_tiles = (int)((N + p->bm * p->cg - 1) / (p->bm * p->cg));
  p->units = (long long)p->n_tiles * p->num_kb;
  skinny_partition(p, max_grid, cfg ? cfg->skinny_grid : 0, cfg ? cfg->skinny_skew_kb : 0);
  return GEMM_OK;
}

// Tiles along M per raster strip: keep the strip's A rows within ~32 MiB of
// L2, so that the strip is re-read from L2 for every tile column it meets.
int raster_group_for(int tile_m, int64_t K, int in_bytes, int tiles_m) {
  const long long strip_bytes = (long long)tile_m * (K > 0 ? K : 1) * in_bytes;
  const long long g = (32ll << 20) / strip_bytes;
  const int group = (int)(g < 1 ? 1 : g);
  return group > tiles_m ? tiles_m : group;
}

void record_launch(const LaunchInfo& li) {
  t_info.path = li.path == 3 ? GEMM_PATH_SKINNY : li.path;
  t_info.grid = li.grid;
  t_info.cluster = li.cluster;
  t_info.block = li.block;
  t_info.tile_m = li.tile_m;
  t_info.tile_n = li.tile_n;
  t_info.stages = li.stages;
  t_info.smem_bytes = li.smem_bytes;
  t_info.kernel = li.kernel;
  t_info.k_parts = li.k_parts;
  t_info.scheduler = li.scheduler;
  t_info.cluster_pref = li.cluster_pref;
  t_info.tail_slices = li.tail_slices > 0 ? li.tail_slices : 1;
}

int run(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
        int64_t ldc, void* D, int64_t ldd, float alpha, float beta, int out_dtype, void* stream_v,
        const gemm_tn_config* cfg, Epilogue epi = Epilogue{nullptr, 0, kActNone}, int in_kind = kInBf16,
        int fp8_format = 0) {
  // Input element: bf16 (2 bytes, 64 per 128-byte stage row) or fp8 (1 byte, 128).
  const int in_bytes = in_kind == kInFp8 ? 1 : 2;
  const int kbe = 128 / in_bytes;
  const CUtensorMapDataType in_dt = in_kind == kInFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  t_error.clear();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  // ---- argument validation
  if (out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F32)
    return fail(GEMM_ERR_INVALID_VALUE, "out_dtype must be 0 (bf16) or 1 (fp32), got %d", out_dtype);
  if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_VALUE, "negative size M=%lld N=%lld K=%lld",
                                           (long long)M, (long long)N, (long long)K);
  int rc = check_config(cfg);
  if (rc != GEMM_OK) return rc;
  const int path_req = cfg ? cfg->path : GEMM_PATH_AUTO;
  const int sched = cfg ? cfg->scheduler : GEMM_SCHED_DEFAULT;
  if (M == 0 || N == 0) return GEMM_OK;
  const bool has_c = (beta != 0.0f);
  const int esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
  rc = check_operands(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, has_c, esize, in_bytes);
  if (rc != GEMM_OK) return rc;

  int dev = 0;
  DeviceState* st = nullptr;
  rc = init_device(&dev, &st);
  if (rc != GEMM_OK) return rc;

  // ---- path
  const int path = path_req == GEMM_PATH_AUTO ? auto_path(M, N, K, in_bytes, st->sms) : path_req;
  if (path == GEMM_PATH_SKINNY && (M > 256 || K == 0))
    return fail(GEMM_ERR_NOT_IMPLEMENTED, "skinny path needs 1 <= M <= 256 and K > 0");

  const CUtensorMapDataType out_dt = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t tmo = timeout_ns(cfg);
  const int fault = cfg ? cfg->test_fault : 0;
  const bool pdl = !(cfg && cfg->disable_pdl);
  LaunchInfo li = {};
  cudaError_t e;

  if (path == GEMM_PATH_SKINNY) {
    const int np = (int)((M + 15) / 16) * 16;
    SkinnyParams p = {};
    if ((rc = skinny_geometry(&p, M, N, K, kbe, st->sms, cfg))) return rc;
    p.kind = in_kind;
    p.a_fmt = fp8_format;
    p.b_fmt = fp8_format;
    const int grid = p.grid;
    p.alpha = alpha; p.beta = beta; p.has_c = has_c; p.epi = epi;
    p.C = C; p.ldc = ldc; p.D = D; p.ldd = ldd; p.out_f32 = out_dtype == GEMM_OUT_F32;
    p.fault = fault; p.timeout_ns = tmo; p.status = st->status;
    p.b_early = cfg && cfg->b_static && pdl ? 1 : 0;
    Workspace* w = nullptr;
    rc = get_workspace(dev, stream, (size_t)grid * p.cg * 2 * p.bm * np, (size_t)p.n_tiles * p.cg * 4, &w);
    if (rc != GEMM_OK) return rc;
    p.partials = w->partials;
    p.counters = w->counters;
    CUtensorMap tA, tB;
    if (p.kg == 1) {
      if ((rc = encode_2d(&tA, in_dt, in_bytes, A, K, M, lda, kbe, np / p.cg, CU_TENSOR_MAP_SWIZZLE_128B, "A")))
        return rc;
      if ((rc = encode_2d(&tB, in_dt, in_bytes, B, K, N, ldb, kbe, p.bm, CU_TENSOR_MAP_SWIZZLE_128B, "B")))
        return rc;
    } else {
      if ((rc = encode_kgroups(&tA, in_dt, in_bytes, A, K, M, lda, kbe, np / p.cg, p.kg, "A"))) return rc;
      if ((rc = encode_kgroups(&tB, in_dt, in_bytes, B, K, N, ldb, kbe, p.bm, p.kg, "B"))) return rc;
    }
    e = launch_skinny(tA, tB, p, pdl, stream, &li);
  } else {
    const int cg = path == GEMM_PATH_2SM ? 2 : 1;
    int tile_m, tile_n, b_rows, epi_r, epi_c;
    tiled_shape(cg, out_dtype == GEMM_OUT_F32, &tile_m, &tile_n, &b_rows, &epi_r, &epi_c);
    TileParams p = {};
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.num_kb = (int)((K + kbe - 1) / kbe);
    p.a_fmt = fp8_format;
    p.b_fmt = fp8_format;
    p.tiles_m = (int)((M + tile_m - 1) / tile_m);
    p.tiles_n = (int)((N + tile_n - 1) / tile_n);
    const long long nt = (long long)p.tiles_m * p.tiles_n;
    if (nt >= ((int64_t)1 << 31)) return fail(GEMM_ERR_INVALID_VALUE, "too many tiles");
    p.num_tiles = (int)nt;
    int group = cfg && cfg->raster_group > 0 ? cfg->raster_group : 0;
    if (group == 0) group = raster_group_for(tile_m, K, in_bytes, p.tiles_m);
    if (group > p.tiles_m) group = p.tiles_m;
    p.raster_group = group;
    p.alpha = alpha; p.beta = beta; p.has_c = has_c; p.epi = epi;
    p.fault = fault; p.timeout_ns = tmo; p.status = st->status;
    p.clc = sched == GEMM_SCHED_CLC ? 1 : 0;
    p.l2_hints = cfg && cfg->l2_hints != 0 ? (cfg->l2_hints < 0 ? 0 : cfg->l2_hints) : kDefaultL2Hints;
    p.cluster_pref = cfg ? cfg->cluster_pref : 0;
    // no split with CLC or a grid override.  A fused epilogue (bias,
    // activation) sits on the finisher's critical path after the hand-off:
    // such calls split only into four parts of at least 32 k-blocks each
    // (measured, bias + tanh-GELU: 256 x 2048 x 8192 42.2 -> 32.9 us, 300 x
    // 1096 x 8192 with SiLU 46.2 -> 32.8 us; but 192 x 4096 x 4096 24.9 ->
    // 29.5 us and two parts of 224 x 8192 x 8192 46.3 -> 46.9 us)
    p.ksplit = p.clc || (cfg && cfg->grid > 0) ? 1 : tiled_parts(p.num_tiles, p.num_kb, st->sms, cg, cfg);
    if ((epi.bias || epi.act) && !(p.ksplit == 4 && p.num_kb >= kFusedSplitMinKb)) p.ksplit = 1;
    if (p.ksplit > p.num_kb) p.ksplit = p.num_kb > 1 ? p.num_kb : 1;  // every part owns a k-block
    if (p.ksplit > 1) {
      // optional: during a capture that would need a larger workspace, run unsplit
      Workspace* w = nullptr;
      rc = get_workspace(dev, stream, (size_t)p.num_tiles * (p.ksplit - 1) * cg * 128 * 256,
                         (size_t)p.num_tiles * cg * 4, &w, true);
      if (rc != GEMM_OK) return rc;
      if (w) {
        p.partials = w->partials;
        p.counters = w->counters;
      } else {
        p.ksplit = 1;
      }
    }
    // slices of the last round (static single launches without a split)
    if (p.ksplit == 1 && !p.clc && !(cfg && cfg->grid > 0) && K > 0)
      tail_slices_plan(p.num_tiles, st->sms / cg, cfg, &p.sub_begin, &p.sub_shift);
    else
      p.sub_begin = p.num_tiles;
    CUtensorMap tA, tB, tC, tD, tBs;
    memset(&tA, 0, sizeof tA);
    memset(&tB, 0, sizeof tB);
    memset(&tC, 0, sizeof tC);
    const CUtensorMapSwizzle out_sw = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (K > 0) {
      if ((rc = encode_2d(&tA, in_dt, in_bytes, A, K, M, lda, kbe, 128, CU_TENSOR_MAP_SWIZZLE_128B, "A")))
        return rc;
      if ((rc = encode_2d(&tB, in_dt, in_bytes, B, K, N, ldb, kbe, b_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                          "B")))
        return rc;
    }
    tBs = tB;
    if (p.sub_shift > 0 && (rc = encode_2d(&tBs, in_dt, in_bytes, B, K, N, ldb, kbe, b_rows >> p.sub_shift,
                                           CU_TENSOR_MAP_SWIZZLE_128B, "B slices")))
      return rc;
    if (has_c && (rc = encode_2d(&tC, out_dt, esize, C, N, M, ldc, epi_c, epi_r, out_sw, "C"))) return rc;
    if ((rc = encode_2d(&tD, out_dt, esize, D, N, M, ldd, epi_c, epi_r, out_sw, "D"))) return rc;
    e = launch_tiled(cg, out_dtype == GEMM_OUT_F32, in_kind, tA, tB, tC, tD, tBs, p, cfg ? cfg->grid : 0, pdl, stream,
                     &li);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(GEMM_ERR_LAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
  }
  record_launch(li);
  return GEMM_OK;
}

// 3D tensor map over a strided batch of row-major matrices.
int encode_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner, uint64_t outer,
              uint64_t batch, uint64_t ld_elems, uint64_t stride_elems, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw, const char* what) {
  cuuint64_t dims[3] = {inner, outer, batch};
  cuuint64_t strides[2] = {ld_elems * (uint64_t)esize, stride_elems * (uint64_t)esize};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled(%s, 3D) failed with %d", what, (int)r);
  return GEMM_OK;
}

// Per-thread staging of one launch's problem list (tensor maps and sizes).
// The launch copies it into the kernel's parameters, so it can be reused as
// soon as the launch call returns.
thread_local GroupList t_list;

int run_grouped(int count, const gemm_problem* probs, float alpha, float beta, int out_dtype, void* stream_v) {
  t_error.clear();
  if (out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F32)
    return fail(GEMM_ERR_INVALID_VALUE, "out_dtype must be 0 (bf16) or 1 (fp32), got %d", out_dtype);
  if (count < 0) return fail(GEMM_ERR_INVALID_VALUE, "negative problem count %d", count);
  if (count == 0) return GEMM_OK;
  if (!probs) return fail(GEMM_ERR_INVALID_VALUE, "problems is NULL");
  const bool has_c = (beta != 0.0f);
  const int esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
  bool any_tall = false, any_work = false;
  for (int i = 0; i < count; ++i) {
    const gemm_problem& q = probs[i];
    if (q.M < 0 || q.N < 0 || q.K < 0)
      return fail(GEMM_ERR_INVALID_VALUE, "problem %d: negative size M=%lld N=%lld K=%lld", i, (long long)q.M,
                  (long long)q.N, (long long)q.K);
    if (q.M == 0 || q.N == 0) continue;
    const int rc = check_operands(q.M, q.N, q.K, q.A, q.lda, q.B, q.ldb, q.C, q.ldc, q.D, q.ldd, has_c, esize, 2);
    if (rc != GEMM_OK) {
      t_error = "problem " + std::to_string(i) + ": " + t_error;
      return rc;
    }
    any_tall = any_tall || q.M > 128;
    any_work = true;
  }
  if (!any_work) return GEMM_OK;
  int dev = 0;
  DeviceState* st = nullptr;
  int rc = init_device(&dev, &st);
  if (rc != GEMM_OK) return rc;

  // One tile shape for the whole list: pair tiles if some problem is taller
  // than 128 rows and the list needs more than one wave of 1-SM tiles, else
  // 1-SM tiles.
  long long small_tiles = 0;
  for (int j = 0; j < count; ++j)
    if (probs[j].M > 0 && probs[j].N > 0) small_tiles += one_sm_tiles(probs[j].M, probs[j].N);
  const int cg = (any_tall && small_tiles > st->sms) ? 2 : 1;
  int tile_m, tile_n, b_rows, epi_r, epi_c;
  tiled_shape(cg, out_dtype == GEMM_OUT_F32, &tile_m, &tile_n, &b_rows, &epi_r, &epi_c);
  const CUtensorMapDataType out_dt = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle out_sw = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  CUtensorMap unused;
  memset(&unused, 0, sizeof unused);
  LaunchInfo li = {};
  int i = 0, launches = 0;
  while (i < count) {
    // the next launch: up to kMaxGroup non-empty problems, below 2^31 tiles
    GroupList& L = t_list;
    memset(&L, 0, sizeof L);
    int n = 0;
    long long tiles = 0;
    for (; i < count && n < kMaxGroup; ++i) {
      const gemm_problem& q = probs[i];
      if (q.M == 0 || q.N == 0) continue;
      GroupProblem& P = L.prob[n];
      P.M = (int)q.M;
      P.N = (int)q.N;
      P.num_kb = (int)((q.K + 63) / 64);
      P.tiles_m = (int)((q.M + tile_m - 1) / tile_m);
      P.tiles_n = (int)((q.N + tile_n - 1) / tile_n);
      if (tiles + (long long)P.tiles_m * P.tiles_n >= (1ll << 31)) {
        if (n == 0) return fail(GEMM_ERR_INVALID_VALUE, "problem %d: too many tiles", i);
        break;
      }
      P.raster_group = raster_group_for(tile_m, q.K, 2, P.tiles_m);
      P.tile_begin = (int)tiles;
      if (q.K > 0) {
        if ((rc = encode_2d(&L.a[n], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q.A, q.K, q.M, q.lda, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B, "A")))
          return rc;
        if ((rc = encode_2d(&L.b[n], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q.B, q.K, q.N, q.ldb, 64, b_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B, "B")))
          return rc;
      }
      if (has_c && (rc = encode_2d(&L.c[n], out_dt, esize, q.C, q.N, q.M, q.ldc, epi_c, epi_r, out_sw, "C")))
        return rc;
      if ((rc = encode_2d(&L.d[n], out_dt, esize, q.D, q.N, q.M, q.ldd, epi_c, epi_r, out_sw, "D"))) return rc;
      tiles += (long long)P.tiles_m * P.tiles_n;
      ++n;
    }
    if (n == 0) break;
    L.count = n;
    TileParams p = {};
    p.M = 1; p.N = 1; p.K = 1; p.num_kb = 1;
    p.tiles_m = 1; p.tiles_n = 1; p.raster_group = 1;
    p.num_tiles = (int)tiles;
    p.alpha = alpha; p.beta = beta; p.has_c = has_c;
    p.timeout_ns = timeout_ns(nullptr); p.status = st->status;
    p.defer_wait = launches > 0 ? 1 : 0;
    const cudaError_t e = launch_tiled_group(cg, out_dtype == GEMM_OUT_F32, kModeList, unused, unused, unused, unused,
                                             &L, p, true, stream, &li);
    ++launches;
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(GEMM_ERR_LAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
    }
  }
  record_launch(li);
  return GEMM_OK;
}

int run_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int64_t sa,
                const void* B, int64_t ldb, int64_t sb, const void* C, int64_t ldc, int64_t sc, void* D, int64_t ldd,
                int64_t sd, float alpha, float beta, int out_dtype, void* stream_v) {
  t_error.clear();
  if (out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F32)
    return fail(GEMM_ERR_INVALID_VALUE, "out_dtype must be 0 (bf16) or 1 (fp32), got %d", out_dtype);
  if (batch < 0 || M < 0 || N < 0 || K < 0)
    return fail(GEMM_ERR_INVALID_VALUE, "negative size batch=%lld M=%lld N=%lld K=%lld", (long long)batch,
                (long long)M, (long long)N, (long long)K);
  if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
  const bool has_c = (beta != 0.0f);
  const int esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
  int rc = check_operands(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, has_c, esize, 2);
  if (rc != GEMM_OK) return rc;
  if (batch >= ((int64_t)1 << 31)) return fail(GEMM_ERR_INVALID_VALUE, "batch must be below 2^31");
  if (batch == 1) {  // the strides are not used; give the maps valid ones
    sa = M * lda;
    sb = N * ldb;
    sc = M * ldc;
    sd = M * ldd;
  }
  if (K > 0 && (sa < M * lda || sb < N * ldb))
    return fail(GEMM_ERR_INVALID_VALUE, "stride_a (%lld) must be >= M*lda and stride_b (%lld) >= N*ldb",
                (long long)sa, (long long)sb);
  if (sd < M * ldd || (has_c && sc < M * ldc))
    return fail(GEMM_ERR_INVALID_VALUE, "stride_d (%lld) must be >= M*ldd and stride_c (%lld) >= M*ldc",
                (long long)sd, (long long)sc);
  if ((K > 0 && ((sa * 2) % 16 || (sb * 2) % 16)) || (sd * esize) % 16 || (has_c && (sc * esize) % 16))
    return fail(GEMM_ERR_MISALIGNED, "batch strides must be multiples of 16 bytes");
  int dev = 0;
  DeviceState* st = nullptr;
  if ((rc = init_device(&dev, &st)) != GEMM_OK) return rc;

  const int cg = (M > 128 && one_sm_tiles(M, N) * batch > st->sms) ? 2 : 1;
  int tile_m, tile_n, b_rows, epi_r, epi_c;
  tiled_shape(cg, out_dtype == GEMM_OUT_F32, &tile_m, &tile_n, &b_rows, &epi_r, &epi_c);
  TileParams p = {};
  p.M = (int)M; p.N = (int)N; p.K = (int)K;
  p.num_kb = (int)((K + 63) / 64);
  p.tiles_m = (int)((M + tile_m - 1) / tile_m);
  p.tiles_n = (int)((N + tile_n - 1) / tile_n);
  const long long nt = (long long)p.tiles_m * p.tiles_n * batch;
  if (nt >= ((int64_t)1 << 31)) return fail(GEMM_ERR_INVALID_VALUE, "too many tiles");
  p.num_tiles = (int)nt;
  p.batch = (int)batch;
  p.raster_group = raster_group_for(tile_m, K, 2, p.tiles_m);
  p.alpha = alpha; p.beta = beta; p.has_c = has_c;
  p.timeout_ns = timeout_ns(nullptr); p.status = st->status;
  const CUtensorMapDataType out_dt = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle out_sw = out_dtype == GEMM_OUT_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap tA, tB, tC, tD;
  memset(&tA, 0, sizeof tA);
  memset(&tB, 0, sizeof tB);
  memset(&tC, 0, sizeof tC);
  if (K > 0) {
    if ((rc = encode_3d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, batch, lda, sa, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B, "A")))
      return rc;
    if ((rc = encode_3d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, batch, ldb, sb, 64, b_rows,
                        CU_TENSOR_MAP_SWIZZLE_128B, "B")))
      return rc;
  }
  if (has_c && (rc = encode_3d(&tC, out_dt, esize, C, N, M, batch, ldc, sc, epi_c, epi_r, out_sw, "C"))) return rc;
  if ((rc = encode_3d(&tD, out_dt, esize, D, N, M, batch, ldd, sd, epi_c, epi_r, out_sw, "D"))) return rc;
  LaunchInfo li = {};
  const cudaError_t e = launch_tiled_group(cg, out_dtype == GEMM_OUT_F32, kModeStrided, tA, tB, tC, tD, nullptr, p,
                                           true, static_cast<cudaStream_t>(stream_v), &li);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(GEMM_ERR_LAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
  }
  record_launch(li);
  return GEMM_OK;
}

}  // namespace

// Sets the text gemm_last_error_string returns on this thread, for entry
// points defined in other files.
void set_error_text(const char* msg) { t_error = msg ? msg : ""; }

// Device address of the current device's status word (the one
// gemm_get_status reads), for entry points defined in other files.
cudaError_t status_word_address(int** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_status);
  if (e == cudaSuccess) *out = static_cast<int*>(p);
  return e;
}

// The wait limit of calls without a config (GEMM_WAIT_TIMEOUT_NS, else 2 s),
// for entry points defined in other files.
uint64_t default_wait_timeout_ns() { return timeout_ns(nullptr); }

// The skinny path's automatic geometry and partition on `sms` SMs, as
// gemm_bf16_tn computes it, for entry points defined in other files.
int skinny_geometry_auto(SkinnyParams* p, int64_t M, int64_t N, int64_t K, int kbe, int sms) {
  return skinny_geometry(p, M, N, K, kbe, sms, nullptr);
}

}  // namespace gtn

extern "C" {

int gemm_bf16_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd, float alpha, float beta, int out_dtype,
                 void* stream) {
  return gtn::run(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream, nullptr);
}

int gemm_bf16_tn_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                    const void* C, int64_t ldc, void* D, int64_t ldd, float alpha, float beta, int out_dtype,
                    void* stream, const gemm_tn_config* cfg) {
  return gtn::run(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream, cfg);
}

int gemm_bf16_tn_grouped(int num_problems, const gemm_problem* problems, float alpha, float beta, int out_dtype,
                         void* stream) {
  return gtn::run_grouped(num_problems, problems, alpha, beta, out_dtype, stream);
}

int gemm_bf16_tn_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int64_t stride_a,
                         const void* B, int64_t ldb, int64_t stride_b, const void* C, int64_t ldc, int64_t stride_c,
                         void* D, int64_t ldd, int64_t stride_d, float alpha, float beta, int out_dtype,
                         void* stream) {
  return gtn::run_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, D, ldd, stride_d,
                          alpha, beta, out_dtype, stream);
}

int gemm_bf16_tn_bias_act(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                          const void* C, int64_t ldc, void* D, int64_t ldd, float alpha, float beta, int out_dtype,
                          const void* bias, int bias_dtype, int activation, void* stream) {
  using namespace gtn;
  if (activation < GEMM_ACT_NONE || activation > GEMM_ACT_SILU)
    return fail(GEMM_ERR_INVALID_VALUE, "unknown activation %d", activation);
  if (bias && bias_dtype != GEMM_OUT_BF16 && bias_dtype != GEMM_OUT_F32)
    return fail(GEMM_ERR_INVALID_VALUE, "bias_dtype must be 0 (bf16) or 1 (fp32), got %d", bias_dtype);
  if (bias && (reinterpret_cast<uintptr_t>(bias) & (bias_dtype == GEMM_OUT_F32 ? 3u : 1u)))
    return fail(GEMM_ERR_MISALIGNED, "bias must be aligned to its element size");
  const Epilogue epi{bias, bias_dtype == GEMM_OUT_F32 ? 1 : 0, activation};
  return run(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream, nullptr, epi);
}

int gemm_fp8_tn_bias_act(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                         int fp8_format, float scale_a, float scale_b, const void* C, int64_t ldc, void* D,
                         int64_t ldd, float alpha, float beta, int out_dtype, const void* bias, int bias_dtype,
                         int activation, void* stream) {
  using namespace gtn;
  if (fp8_format != GEMM_FP8_E4M3 && fp8_format != GEMM_FP8_E5M2)
    return fail(GEMM_ERR_INVALID_VALUE, "fp8_format must be 0 (e4m3) or 1 (e5m2), got %d", fp8_format);
  if (activation < GEMM_ACT_NONE || activation > GEMM_ACT_SILU)
    return fail(GEMM_ERR_INVALID_VALUE, "unknown activation %d", activation);
  if (bias && bias_dtype != GEMM_OUT_BF16 && bias_dtype != GEMM_OUT_F32)
    return fail(GEMM_ERR_INVALID_VALUE, "bias_dtype must be 0 (bf16) or 1 (fp32), got %d", bias_dtype);
  if (bias && (reinterpret_cast<uintptr_t>(bias) & (bias_dtype == GEMM_OUT_F32 ? 3u : 1u)))
    return fail(GEMM_ERR_MISALIGNED, "bias must be aligned to its element size");
  const Epilogue epi{bias, bias_dtype == GEMM_OUT_F32 ? 1 : 0, activation};
  return run(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha * scale_a * scale_b, beta, out_dtype, stream, nullptr,
             epi, kInFp8, fp8_format);
}

int gemm_fp8_tn_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   int fp8_format, float scale_a, float scale_b, const void* C, int64_t ldc, void* D, int64_t ldd,
                   float alpha, float beta, int out_dtype, void* stream, const gemm_tn_config* cfg) {
  using namespace gtn;
  if (fp8_format != GEMM_FP8_E4M3 && fp8_format != GEMM_FP8_E5M2)
    return fail(GEMM_ERR_INVALID_VALUE, "fp8_format must be 0 (e4m3) or 1 (e5m2), got %d", fp8_format);
  return run(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha * scale_a * scale_b, beta, out_dtype, stream, cfg,
             Epilogue{nullptr, 0, kActNone}, kInFp8, fp8_format);
}

int gemm_fp8_tn(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                int fp8_format, float scale_a, float scale_b, const void* C, int64_t ldc, void* D, int64_t ldd,
                float alpha, float beta, int out_dtype, void* stream) {
  return gemm_fp8_tn_ex(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C, ldc, D, ldd, alpha, beta,
                        out_dtype, stream, nullptr);
}

int gemm_plan(int64_t M, int64_t N, int64_t K, int fp8_inputs, int num_sms, const gemm_tn_config* cfg,
              gemm_plan_info* out) {
  using namespace gtn;
  t_error.clear();
  if (!out) return fail(GEMM_ERR_INVALID_VALUE, "out is NULL");
  *out = gemm_plan_info{};
  if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_VALUE, "negative size");
  if (num_sms < 1) return fail(GEMM_ERR_INVALID_VALUE, "num_sms must be at least 1, got %d", num_sms);
  if (fp8_inputs != 0 && fp8_inputs != 1) return fail(GEMM_ERR_INVALID_VALUE, "fp8_inputs must be 0 or 1");
  int rc = check_config(cfg);
  if (rc != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  const int in_bytes = fp8_inputs ? 1 : 2;
  const int path_req = cfg ? cfg->path : GEMM_PATH_AUTO;
  const int path = path_req == GEMM_PATH_AUTO ? auto_path(M, N, K, in_bytes, num_sms) : path_req;
  if (path == GEMM_PATH_SKINNY && (M > 256 || K == 0))
    return fail(GEMM_ERR_NOT_IMPLEMENTED, "skinny path needs 1 <= M <= 256 and K > 0");
  out->path = path;
  out->tail_slices = 1;
  if (path == GEMM_PATH_SKINNY) {
    SkinnyParams p = {};
    if ((rc = skinny_geometry(&p, M, N, K, 128 / in_bytes, num_sms, cfg))) return rc;
    out->tile_m = p.bm * p.cg;
    out->tile_n = p.np;
    out->skinny_kgroup = p.kg;
    out->skinny_stages = p.stages;
    out->skinny_grid = p.grid * p.cg;
    out->k_parts = p.split;
    out->skinny_skew = p.skew;
  } else {
    int tm, tn, br, er, ec;
    tiled_shape(path == GEMM_PATH_2SM ? 2 : 1, 0, &tm, &tn, &br, &er, &ec);
    out->tile_m = tm;
    out->tile_n = tn;
    const long long tiles = ((M + tm - 1) / tm) * ((N + tn - 1) / tn);
    const bool clc = cfg && cfg->scheduler == GEMM_SCHED_CLC;
    const int cg = path == GEMM_PATH_2SM ? 2 : 1;
    out->k_parts = clc || (cfg && cfg->grid > 0) || K == 0
                       ? 1 : tiled_parts(tiles, (int)((K + 128 / in_bytes - 1) / (128 / in_bytes)), num_sms, cg, cfg);
    out->tail_slices = 1;
    if (out->k_parts == 1 && !clc && !(cfg && cfg->grid > 0) && K > 0) {
      int begin = 0, shift = 0;
      tail_slices_plan(tiles, num_sms / cg, cfg, &begin, &shift);
      out->tail_slices = 1 << shift;
    }
  }
  return GEMM_OK;
}

int gemm_get_status(void* stream) {
  using namespace gtn;
  t_error.clear();
  int dev = 0;
  DeviceState* st = nullptr;
  int rc = init_device(&dev, &st);
  if (rc != GEMM_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  int h[kStatusWords] = {0, 0};
  e = cudaMemcpy(h, st->status, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (h[0] == 0) return GEMM_OK;
  int z[kStatusWords] = {0, 0};
  e = cudaMemcpy(st->status, z, sizeof z, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  {
    // An aborted skinny kernel can leave arrival counters set: clear them.
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& kv : g_ws)
      if (kv.first.first == dev && kv.second.counters)
        cudaMemset(kv.second.counters, 0, kv.second.counter_ints * sizeof(int));
  }
  cudaDeviceSynchronize();
  t_last_detail = h[1];
  return fail(h[0], "device wait timed out (role %d, block %d)", h[1] >> 24, h[1] & 0xFFFFFF);
}

int gemm_get_status_detail(void) { return gtn::t_last_detail; }

const char* gemm_last_error_string(void) { return gtn::t_error.c_str(); }

int gemm_last_launch_info(gemm_launch_info* out) {
  if (!out) return GEMM_ERR_INVALID_VALUE;
  *out = gtn::t_info;
  return GEMM_OK;
}

void gemm_shutdown(void) {
  using namespace gtn;
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_ws) {
    cudaSetDevice(kv.first.first);
    if (kv.second.partials) cudaFree(kv.second.partials);
    if (kv.second.counters) cudaFree(kv.second.counters);
  }
  g_ws.clear();
  cudaSetDevice(cur);
}

int gemm_version(void) { return 100; }

}  // extern "C"
