// gemm_bf16_tn_skinny_noalloc: the skinny (M <= 64) path with its scratch
// memory in a fixed device array instead of a library allocation.
//
// Who needs it: callers that must not allocate device memory at call time —
// code that runs under a memory budget fixed up front (an inference server
// that reserves all of HBM for its own pool), code on a latency-critical
// path where cudaMalloc's implicit device synchronisation is unacceptable,
// and plug-ins whose host framework owns every allocation.  The regular
// entry point allocates the skinny path's workspace on first use per
// (device, stream); this one never calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// The scratch array below holds the fp32 partial sums of tiles split
// between CTAs and their arrival counters.  It is part of the library image:
// every device that loads the library keeps it (about 10 MiB) until the
// process exits.  All calls on a device share it, so two calls of this
// entry point whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it; calls in one stream are ordered and do
// not.  The counters must start at zero, so each call clears them on its
// stream before the kernel runs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/gemm_tn.h"
#include "kernels.h"

namespace gtn {
namespace {

// Limits of the fixed scratch (checked on every call).
constexpr int kNaMaxM = 64;          // tokens (the skinny path's limit)
constexpr int kNaMaxGrid = 160;      // CTAs; one per SM on a 152-SM GB300
constexpr int kNaMaxTiles = 1024;    // 128-row tiles of B: N <= 131072
constexpr size_t kNaPartialFloats = (size_t)kNaMaxGrid * 2 * 128 * kNaMaxM;  // 10 MiB
constexpr size_t kNaCounterInts = (size_t)kNaMaxTiles * 4;
constexpr size_t kNaScratchBytes = kNaPartialFloats * 4 + kNaCounterInts * 4;

// Zero-initialised when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

constexpr int kMaxDevices = 64;

struct NaDevice {
  bool ready = false;
  int sms = 0;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int* status = nullptr;             // device status word (gemm_get_status)
};

std::mutex g_na_mu;
NaDevice g_na[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_na_encode = nullptr;

// Per-device set-up on the first call with that device current: look up the
// scratch array's device address (the host-side symbol is only a stand-in)
// and the status word.  Touches no allocator.
int na_setup(int dev, NaDevice** out) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  NaDevice& d = g_na[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3)) return GEMM_ERR_UNSUPPORTED_DEVICE;
    d.sms = prop.multiProcessorCount;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
    d.scratch = static_cast<unsigned char*>(p);
    if (status_word_address(&d.status) != cudaSuccess) return GEMM_ERR_CUDA;
    if (!g_na_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return GEMM_ERR_CUDA;
      g_na_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return GEMM_OK;
}

// bf16 operand map with 64-element k-blocks: 2D (kg = 1), or the 3D view
// {k in block, row, k-block} that loads kg k-blocks per box (K a multiple of 64).
int na_encode(CUtensorMap* m, const void* base, uint64_t K, uint64_t outer, uint64_t ld, uint32_t box_outer, int kg) {
  CUresult r;
  if (kg == 1) {
    cuuint64_t dims[2] = {K, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64, box_outer};
    cuuint32_t estr[2] = {1, 1};
    r = g_na_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, outer, K / 64};
    cuuint64_t strides[2] = {ld * 2, 128};
    cuuint32_t box[3] = {64, box_outer, (cuuint32_t)kg};
    cuuint32_t estr[3] = {1, 1, 1};
    r = g_na_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

int na_fail(int code, const char* msg) {
  set_error_text(msg);
  return code;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gtn

extern "C" int gemm_bf16_tn_skinny_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                           int64_t ldb, const void* C, int64_t ldc, void* D, int64_t ldd, float alpha,
                                           float beta, int out_dtype, void* stream_v) {
  using namespace gtn;
  set_error_text("");
  const bool has_c = beta != 0.0f;
  const int esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
  if (out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F32) return na_fail(GEMM_ERR_INVALID_VALUE, "bad out_dtype");
  if (M < 1 || M > kNaMaxM) return na_fail(GEMM_ERR_INVALID_VALUE, "no-alloc path needs 1 <= M <= 64");
  if (N < 1 || N > (int64_t)kNaMaxTiles * 128)
    return na_fail(GEMM_ERR_INVALID_VALUE, "no-alloc path needs 1 <= N <= 131072 (fixed scratch size)");
  if (K < 1 || K >= ((int64_t)1 << 31)) return na_fail(GEMM_ERR_INVALID_VALUE, "no-alloc path needs 1 <= K < 2^31");
  if (!A || !B || !D || (has_c && !C)) return na_fail(GEMM_ERR_INVALID_VALUE, "NULL operand");
  if (lda < K || ldb < K || ldd < N || (has_c && ldc < N))
    return na_fail(GEMM_ERR_INVALID_VALUE, "leading dimension smaller than the matrix");
  if (!al16(A) || !al16(B) || !al16(D) || (has_c && !al16(C)) || (lda * 2) % 16 || (ldb * 2) % 16 ||
      (ldd * esize) % 16 || (has_c && (ldc * esize) % 16))
    return na_fail(GEMM_ERR_MISALIGNED, "pointers must be 16-byte aligned and rows multiples of 16 bytes");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return na_fail(GEMM_ERR_CUDA, "no current device");
  NaDevice* d = nullptr;
  int rc = na_setup(dev, &d);
  if (rc != GEMM_OK) return na_fail(rc, "device set-up failed (needs sm_103)");

  // The same geometry and partition as gemm_bf16_tn's skinny path, on at
  // most kNaMaxGrid SMs; then every bound the fixed scratch rests on is
  // checked before anything is launched.
  SkinnyParams p = {};
  const int sms = d->sms < kNaMaxGrid ? d->sms : kNaMaxGrid;
  rc = skinny_geometry_auto(&p, M, N, K, 64, sms);
  if (rc != GEMM_OK) return rc;
  if (p.grid < 1 || p.grid > kNaMaxGrid || (size_t)p.n_tiles * 4 > kNaCounterInts ||
      (size_t)p.grid * 2 * p.bm * p.np > kNaPartialFloats)
    return na_fail(GEMM_ERR_INVALID_VALUE, "shape needs more scratch than the no-alloc path holds");
  p.alpha = alpha;
  p.beta = beta;
  p.has_c = has_c;
  p.C = C;
  p.ldc = ldc;
  p.D = D;
  p.ldd = ldd;
  p.out_f32 = out_dtype == GEMM_OUT_F32;
  p.partials = reinterpret_cast<float*>(d->scratch);
  p.counters = reinterpret_cast<int*>(d->scratch + kNaPartialFloats * 4);
  p.fault = 0;
  p.timeout_ns = default_wait_timeout_ns();
  p.status = d->status;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  // The arrival counters must start at zero.
  if (cudaMemsetAsync(p.counters, 0, (size_t)p.n_tiles * 4 * sizeof(int), stream) != cudaSuccess)
    return na_fail(GEMM_ERR_CUDA, "clearing the counters failed");
  CUtensorMap tA, tB;
  if (na_encode(&tA, A, K, M, lda, p.np, p.kg) != GEMM_OK || na_encode(&tB, B, K, N, ldb, (uint32_t)p.bm, p.kg) != GEMM_OK)
    return na_fail(GEMM_ERR_LAUNCH, "tensor map encoding failed");
  LaunchInfo li = {};
  if (launch_skinny(tA, tB, p, false, stream, &li) != cudaSuccess) {
    cudaGetLastError();
    return na_fail(GEMM_ERR_LAUNCH, "kernel launch failed");
  }
  return GEMM_OK;
}
