// Measurement kernels: the read ceiling of the skinny kernel's operand
// stream (gemm_stream_read) and the tcgen05.mma rate at the skinny path's
// shapes (gemm_mma_rate).
//
// gemm_stream_read: the read ceiling of the skinny kernel's operand stream.
//
// The Ampere-to-Hopper page (section "not reaching peak") judges a kernel
// against ceilings measured on the same box rather than against datasheet
// numbers.  For the HBM-bound decode GEMM the relevant ceiling is not a
// device-to-device copy (which also writes) but a stream of the same TMA
// boxes into the same shared-memory ring with nothing else to do: every CTA
// has one thread that keeps `stages` boxes in flight and re-issues a stage
// as soon as its bytes have landed.  The data is never consumed.  The time
// of one launch over the decode's weight matrix is what the GEMM could take
// if its MMAs, token loads and epilogue cost nothing.
//
// Work order matches the skinny kernel: the matrix is cut into tiles of
// box_rows rows; within a tile the unit is a group of kgroup 128-byte
// k-chunks; CTA c streams the contiguous unit range
// [c * units / grid, (c + 1) * units / grid).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/gemm_tn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gtn {
namespace {

constexpr int kSrRing = 216 * 1024;   // ring bytes per CTA (the skinny kernel's)
constexpr int kSrMaxStages = 64;

struct StreamParams {
  long long units;      // tiles * groups
  long long groups;     // k-groups per tile
  int box_rows, kgroup, stages, stage_bytes;
  uint64_t timeout_ns;
  int* status;
};

__global__ void __launch_bounds__(32, 1) gemm_stream_read_kernel(const __grid_constant__ CUtensorMap tm,
                                                                 const StreamParams p) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x != 0) return;
  const uint32_t base = smem_u32(smem);
  const uint32_t bar0 = base + p.stages * p.stage_bytes;
  for (int s = 0; s < p.stages; ++s) mbar_init(bar0 + 8 * s, 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  const long long b = (long long)blockIdx.x * p.units / gridDim.x;
  const long long e = (long long)(blockIdx.x + 1) * p.units / gridDim.x;
  auto issue = [&](long long u, int s) {
    const int tile = (int)(u / p.groups), grp = (int)(u % p.groups);
    const uint32_t bar = bar0 + 8 * s;
    mbar_arrive_expect_tx(bar, (uint32_t)p.stage_bytes);
    tma_load_3d(base + s * p.stage_bytes, &tm, 0, tile * p.box_rows, grp * p.kgroup, bar);
  };
  long long issued = b;
  for (int s = 0; s < p.stages && issued < e; ++s) issue(issued++, s);
  bool failed = false;
  for (long long u = b; u < issued; ++u) {
    const int s = (int)((u - b) % p.stages);
    const uint32_t par = (uint32_t)(((u - b) / p.stages) & 1);
    const uint64_t t0 = globaltimer();
    bool ok = true;
    while (!mbar_try_wait(bar0 + 8 * s, par)) {
      if (globaltimer() - t0 > p.timeout_ns) {
        ok = false;
        break;
      }
    }
    if (!ok && !failed) {
      failed = true;
      if (atomicCAS(p.status, 0, GEMM_ERR_TIMEOUT) == 0) atomicExch(p.status + 1, (kRoleProducer << 24) | (int)blockIdx.x);
    }
    // After a failure nothing new is issued; the loop still waits (bounded)
    // once for every copy already in flight so that none lands after exit.
    if (!failed && issued < e) issue(issued++, s);
  }
}

// One CTA (CG = 1) or CTA pair (CG = 2) issues `reps` groups of four
// tcgen05.mma (K = 16 bf16 or 32 fp8 each, walking one 128-byte K atom) on
// zeroed shared-memory operands: MMA M = 128 per CTA, N = n (split between
// the pair's CTAs for CG = 2), accumulating into TMEM, then commits and waits
// (bounded).  out[0] = ns from the first issue to completion, out[1] = ns of
// issue alone.  The operands' values do not matter for the timing.
constexpr int kRateStages = 3;

template <int CG, int KIND>
__global__ void __launch_bounds__(64, 1) gemm_mma_rate_kernel(int n, int reps, uint64_t timeout_ns, int* status,
                                                              unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0;
  const int nb = n / CG;                                 // B rows held by this CTA
  const uint32_t sA = smem_u32(smem);                    // stages x 128 rows x 128 B
  const uint32_t sB = sA + kRateStages * 16384;          // stages x nb rows x 128 B
  for (int i = threadIdx.x; i < kRateStages * (16384 + nb * 128) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) tmem_alloc<CG>(smem_u32(&tslot), 256);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    bool ok = true;
    if (rank == 0) {
      const uint32_t idesc = KIND == kKindF16 ? instr_desc_bf16_f32(128 * CG, (uint32_t)n)
                                              : instr_desc_f32acc(128 * CG, (uint32_t)n, 0, 0);
      const unsigned long long t0 = globaltimer();
      for (int r = 0; r < reps; ++r) {
        const int st = r % kRateStages;
        const uint64_t a0 = smem_desc_sw128(sA + st * 16384), b0 = smem_desc_sw128(sB + st * nb * 128);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_issue<CG, KIND>(tmem, a0 + 2 * k, b0 + 2 * k, idesc, (r | k) ? 1u : 0u);
      }
      if constexpr (CG == 1) mma_commit(smem_u32(&bar));
      else mma_commit_pair(smem_u32(&bar), 0x3);
      const unsigned long long t1 = globaltimer();
      ok = false;
      while (globaltimer() - t1 < timeout_ns)
        if (mbar_try_wait(smem_u32(&bar), 0)) { ok = true; break; }
      const unsigned long long t2 = globaltimer();
      if (blockIdx.x == 0) {
        out[0] = t2 - t0;
        out[1] = t1 - t0;
      }
    } else {
      const unsigned long long t1 = globaltimer();
      ok = false;
      while (globaltimer() - t1 < timeout_ns)
        if (mbar_try_wait_cluster(smem_u32(&bar), 0)) { ok = true; break; }
    }
    if (!ok && atomicCAS(status, 0, GEMM_ERR_TIMEOUT) == 0) atomicExch(status + 1, (kRoleMma << 24) | (int)blockIdx.x);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, 256);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_sr_mu;
EncodeTiledFn g_sr_encode = nullptr;

int sr_fail(int code, const char* msg) {
  set_error_text(msg);
  return code;
}

}  // namespace
}  // namespace gtn

extern "C" int gemm_stream_read(const void* src, int64_t rows, int64_t row_bytes, int box_rows, int kgroup, int grid,
                                void* stream_v) {
  using namespace gtn;
  set_error_text("");
  if (!src || (reinterpret_cast<uintptr_t>(src) & 15u)) return sr_fail(GEMM_ERR_MISALIGNED, "src must be 16-byte aligned");
  if (!(box_rows == 32 || box_rows == 64 || box_rows == 128 || box_rows == 256))
    return sr_fail(GEMM_ERR_INVALID_VALUE, "box_rows must be 32, 64, 128 or 256");
  if (!(kgroup == 1 || kgroup == 2 || kgroup == 4)) return sr_fail(GEMM_ERR_INVALID_VALUE, "kgroup must be 1, 2 or 4");
  if (rows < box_rows || rows % box_rows || rows >= ((int64_t)1 << 31))
    return sr_fail(GEMM_ERR_INVALID_VALUE, "rows must be a positive multiple of box_rows below 2^31");
  if (row_bytes < 128 * kgroup || row_bytes % (128 * kgroup) || row_bytes >= ((int64_t)1 << 31))
    return sr_fail(GEMM_ERR_INVALID_VALUE, "row_bytes must be a positive multiple of 128 * kgroup below 2^31");
  if (grid < 0) return sr_fail(GEMM_ERR_INVALID_VALUE, "grid must be >= 0");
  const int stage_bytes = box_rows * 128 * kgroup;
  int stages = kSrRing / stage_bytes;
  if (stages > kSrMaxStages) stages = kSrMaxStages;
  if (stages < 2) return sr_fail(GEMM_ERR_INVALID_VALUE, "box too large for a two-stage ring");

  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return sr_fail(GEMM_ERR_CUDA, "no current device");
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return sr_fail(GEMM_ERR_CUDA, "device query failed");
  if (!(major == 10 && minor == 3)) return sr_fail(GEMM_ERR_UNSUPPORTED_DEVICE, "needs sm_103");
  int* status = nullptr;
  if (status_word_address(&status) != cudaSuccess) return sr_fail(GEMM_ERR_CUDA, "status word lookup failed");
  {
    std::lock_guard<std::mutex> lk(g_sr_mu);
    if (!g_sr_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return sr_fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled not available");
      g_sr_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  // 3D view {byte in chunk, row, 128-byte chunk}: one box = box_rows rows x
  // kgroup consecutive chunks, each chunk landing as its own 128-byte-swizzled
  // block, as the skinny kernel loads its weights.
  CUtensorMap tm;
  cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128)};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
  cuuint32_t box[3] = {128, (cuuint32_t)box_rows, (cuuint32_t)kgroup};
  cuuint32_t estr[3] = {1, 1, 1};
  if (g_sr_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(src), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return sr_fail(GEMM_ERR_LAUNCH, "tensor map encoding failed");

  StreamParams p = {};
  p.groups = row_bytes / 128 / kgroup;
  p.units = (rows / box_rows) * p.groups;
  p.box_rows = box_rows;
  p.kgroup = kgroup;
  p.stages = stages;
  p.stage_bytes = stage_bytes;
  p.timeout_ns = default_wait_timeout_ns();
  p.status = status;
  long long g = grid > 0 ? grid : sms;
  if (g > p.units) g = p.units;
  const int smem = 1024 + stages * stage_bytes + 8 * stages;
  if (cudaFuncSetAttribute(gemm_stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return sr_fail(GEMM_ERR_LAUNCH, "shared-memory attribute rejected");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream_v);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemm_stream_read_kernel, tm, p) != cudaSuccess) {
    cudaGetLastError();
    return sr_fail(GEMM_ERR_LAUNCH, "kernel launch failed");
  }
  return GEMM_OK;
}

extern "C" int gemm_mma_rate(int n, int cta_group, int fp8, int reps, int grid, unsigned long long* out_ns,
                             void* stream_v) {
  using namespace gtn;
  set_error_text("");
  if (cta_group != 1 && cta_group != 2) return sr_fail(GEMM_ERR_INVALID_VALUE, "cta_group must be 1 or 2");
  if (n < 16 || n > 256 || n % 16) return sr_fail(GEMM_ERR_INVALID_VALUE, "n must be a multiple of 16 in [16, 256]");
  if (reps < 1 || reps > (1 << 24)) return sr_fail(GEMM_ERR_INVALID_VALUE, "reps must be in [1, 2^24]");
  if (grid < 1 || grid > 1024 || grid % cta_group) return sr_fail(GEMM_ERR_INVALID_VALUE, "bad grid");
  if (!out_ns || (reinterpret_cast<uintptr_t>(out_ns) & 7u)) return sr_fail(GEMM_ERR_MISALIGNED, "out_ns");
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return sr_fail(GEMM_ERR_CUDA, "device query failed");
  if (!(major == 10 && minor == 3)) return sr_fail(GEMM_ERR_UNSUPPORTED_DEVICE, "needs sm_103");
  int* status = nullptr;
  if (status_word_address(&status) != cudaSuccess) return sr_fail(GEMM_ERR_CUDA, "status word lookup failed");
  const int smem = 1024 + kRateStages * (16384 + n / cta_group * 128);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(64);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream_v);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cta_group;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint64_t tmo = default_wait_timeout_ns();
  cudaError_t e;
#define GTN_RATE(CGV, KV)                                                                              \
  ((e = cudaFuncSetAttribute(gemm_mma_rate_kernel<CGV, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) \
       == cudaSuccess                                                                                  \
       ? cudaLaunchKernelEx(&cfg, gemm_mma_rate_kernel<CGV, KV>, n, reps, tmo, status, out_ns)           \
       : e)
  if (cta_group == 1) e = fp8 ? GTN_RATE(1, kKindF8F6F4) : GTN_RATE(1, kKindF16);
  else e = fp8 ? GTN_RATE(2, kKindF8F6F4) : GTN_RATE(2, kKindF16);
#undef GTN_RATE
  if (e != cudaSuccess) {
    cudaGetLastError();
    return sr_fail(GEMM_ERR_LAUNCH, "kernel launch failed");
  }
  return GEMM_OK;
}
