// Internal interface between the C-ABI layer (gemm_api.cu) and the kernel
// translation units.  Not installed; the public surface is include/gemm_tn.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gtn {

// Input kinds (match the tcgen05.mma kinds in ptx.cuh).
constexpr int kInBf16 = 0;
constexpr int kInFp8 = 1;

// Device status word: [0] = first error code (0 = none), [1] = detail
// (role << 24 | block index) of the wait that gave up.
constexpr int kStatusWords = 2;

enum Role : int { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleFixup = 4 };

// L2 eviction-priority hints of the tiled kernels' copies (TileParams.l2_hints).
constexpr int kL2HintAEvictLast = 1, kL2HintBEvictFirst = 2, kL2HintDEvictFirst = 4;

// Test-only fault injection bits.
constexpr int kFaultSkipTmaOnce = 1;

// Activation codes (same values as gemm_activation in gemm_tn.h).
constexpr int kActNone = 0, kActRelu = 1, kActGelu = 2, kActGeluTanh = 3, kActSilu = 4;

// Fused epilogue: D = act(alpha * acc + beta * C + bias[n]).
struct Epilogue {
  const void* bias;    // N values (bf16 or fp32) or nullptr
  int bias_f32;
  int act;             // kAct*
};

// Problem sources of the tiled kernel: one GEMM; a list of up to kMaxGroup
// GEMMs of any shapes, each with its own tensor maps (kernel parameters); or
// a strided batch of equal GEMMs read through 3D tensor maps (the third
// coordinate is the batch index).
constexpr int kModeSingle = 0, kModeList = 1, kModeStrided = 2;
constexpr int kMaxGroup = 56;   // per launch: 56 x 4 tensor maps fill most of the 32 KB of kernel parameters

struct GroupProblem {
  int M, N, num_kb;
  int tiles_m, tiles_n, raster_group;
  int tile_begin;      // first tile of this problem in the launch's tile order
  int pad;
};

struct GroupList {
  CUtensorMap a[kMaxGroup], b[kMaxGroup], c[kMaxGroup], d[kMaxGroup];
  GroupProblem prob[kMaxGroup];
  int count;
};

struct NoGroup {
  int unused;
};

struct TileParams {
  int M, N, K;
  int num_kb;          // ceil(K / 64)
  int tiles_m, tiles_n, num_tiles;
  int raster_group;    // tiles along M per grouped-raster strip
  float alpha, beta;
  int has_c;           // beta != 0
  int a_fmt, b_fmt;    // fp8 inputs: kind::f8f6f4 format codes (0 = e4m3, 1 = e5m2)
  int clc;             // 1 = one CTA (pair) launched per tile, work taken over by cluster launch control
  int batch;           // strided batch: number of problems (tiles = batch * tiles_m * tiles_n)
  int defer_wait;      // 1 = later launch of one grouped call: wait for the previous launch at the end, not
                       // the start (the launches' problems are independent; see the kernel)
  Epilogue epi;
  int l2_hints;        // kL2Hint* bits (single problems only)
  int cluster_pref;    // host only: preferred cluster size (4 or 8 CTAs) of a static pair launch, 0 = none
  int fault;           // kFault* bits (tests only)
  uint64_t timeout_ns;
  int* status;
  // k-split of single-problem launches (static schedule, one unit per
  // cluster): unit u is tile u % num_tiles, part ksplit - 1 - u / num_tiles
  // (so the part that finishes a tile has the highest cluster ids), k-blocks
  // [part * num_kb / ksplit, (part + 1) * num_kb / ksplit).  Parts > 0 write
  // fp32 partials; part 0 adds them in part order.
  int ksplit;          // parts per tile (1 = no split)
  int num_units;       // num_tiles * ksplit, or with slices sub_begin + (num_tiles - sub_begin) << sub_shift
  // Slices of the last, partial round (single problems, static schedule, no
  // k-split): unit u >= sub_begin is slice (u - sub_begin) % 2^sub_shift, of
  // width 256 >> sub_shift columns, of tile sub_begin + (u - sub_begin) >>
  // sub_shift, so that the round's r tiles occupy r << sub_shift clusters.
  int sub_begin;       // first slice unit (num_units when no tile is sliced)
  int sub_shift;       // log2 of the slices per tile: 0, 1 or 2
  float* partials;     // num_tiles * (ksplit - 1) * cta_group * 128 * 256 floats
  int* counters;       // num_tiles * cta_group * 4, zero between calls
};

struct SkinnyParams {
  int M, N, K;
  int np;              // M rounded up to 16 (MMA N), 16..64
  int num_kb;          // k-groups per tile: ceil(ceil(K / k-block) / kg)
  int kg;              // k-blocks per ring stage (1, 2 or 4); > 1 loads through 3D tensor maps
                       //    {k in block, row, k-block} with one box of kg k-blocks per operand
  int n_tiles;         // ceil(N / bm)
  long long units;     // n_tiles * num_kb (one unit = one k-group of one tile)
  int grid;            // CTAs; each owns a contiguous range of units
  int split;           // 0: stream-K ranges over the grid; s >= 2: every tile in s parts,
                       //    CTA c holds part c / n_tiles of tile c % n_tiles
  int skew;            // split mode: k-groups moved from the last part to part 0
  int b_early;         // 1 = B is not written by anything still running: its first ring is loaded
                       //    before the dependency wait on the previous kernel
  int stages;
  float alpha, beta;
  int has_c;
  const void* C; long long ldc;
  void* D; long long ldd;
  int out_f32;
  int bm;              // rows of B per tile (MMA M): 128, or 64; per CTA in the pair form
  int cg;              // 1, or 2 = pair form: clusters of two CTAs on tiles of 2 * bm rows (MMA M = 256),
                       //    each CTA holding np / 2 token rows; grid, split and units count pairs
  int kind;            // kKindF16 (bf16 inputs) or kKindF8F6F4 (fp8 inputs)
  int a_fmt, b_fmt;    // fp8 format codes
  Epilogue epi;
  float* partials;     // grid * 2 slots * 128 * np floats
  int* counters;       // 4 per n-tile (one per epilogue warp), zero between calls
  int fault;
  uint64_t timeout_ns;
  int* status;
};

struct LaunchInfo {
  int path;            // 1 = 1-SM tiled, 2 = 2-SM tiled, 3 = skinny
  int grid, cluster, block;
  int tile_m, tile_n, stages;
  int smem_bytes;
  const char* kernel;
  int scheduler;       // 1 = static persistent, 2 = cluster launch control (tiled paths)
  int k_parts;         // k-parts per tile (tiled split; skinny equal split), 0 = skinny stream-K
  int cluster_pref;    // preferred cluster size requested at launch (0 = none)
  int tail_slices;     // tiled: slices per tile of the last round (1 = none)
};

// Tiled persistent kernels (1-SM or 2-SM).  Returns a cudaError_t.  `pdl`
// launches with programmatic stream serialisation: the kernel's set-up may
// overlap the previous kernel on the stream; it waits for that kernel's
// completion (griddepcontrol.wait) before touching global memory.
// `tmBs` is B with boxes of b_rows_per_cta >> p.sub_shift rows, for the
// slices of the last round (ignored when p.sub_begin >= p.num_units).
cudaError_t launch_tiled(int cta_group, int out_f32, int kind, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmC, const CUtensorMap& tmD, const CUtensorMap& tmBs, TileParams p,
                         int grid_override, bool pdl, cudaStream_t stream, LaunchInfo* info);


// The same kernels over a list of problems (bf16 inputs; `list` holds the
// per-problem tensor maps and sizes, p.num_tiles their total tile count) or
// over a strided batch (3D tensor maps in tmA..tmD, p.batch problems).
cudaError_t launch_tiled_group(int cta_group, int out_f32, int mode, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmD,
                               const GroupList* list, TileParams p, bool pdl, cudaStream_t stream, LaunchInfo* info);

// Tile shape of the tiled kernels for a CTA group size (for host set-up).
void tiled_shape(int cta_group, int out_f32, int* tile_m, int* tile_n, int* b_rows_per_cta,
                 int* epi_rows, int* epi_cols);

// Skinny (M <= 64) swap-AB stream-K kernel.
cudaError_t launch_skinny(const CUtensorMap& tmA, const CUtensorMap& tmB, SkinnyParams p, bool pdl,
                          cudaStream_t stream, LaunchInfo* info);

// Device address of the current device's status word (gemm_api.cu).
cudaError_t status_word_address(int** out);
// Text returned by gemm_last_error_string on this thread (gemm_api.cu).
void set_error_text(const char* msg);
// Wait limit of calls without a config: GEMM_WAIT_TIMEOUT_NS, else 2 s (gemm_api.cu).
uint64_t default_wait_timeout_ns();
// The skinny path's automatic geometry and partition (tile rows, k-group,
// tiles, units, grid, split, skew, stages) for M x N x K with kbe elements per
// k-block on `sms` SMs; GEMM_OK or a gemm_status code (gemm_api.cu).
int skinny_geometry_auto(SkinnyParams* p, int64_t M, int64_t N, int64_t K, int kbe, int sms);

// Largest co-resident grid for the skinny kernel at this np.
int skinny_max_grid(int np, int num_sms);
// Work partition of the skinny kernel: fills p->grid, p->split and p->skew
// from p->n_tiles and p->num_kb.  grid_override > 0 forces a stream-K grid;
// skew_kb: 0 = default, > 0 = that many k-blocks, < 0 = none.
void skinny_partition(SkinnyParams* p, int num_sms, int grid_override, int skew_kb);
int skinny_stages(int np, int bm, int kg);
// k-blocks per skinny ring stage for K (kbe elements per k-block): kg_req if
// non-zero, else the largest of 4, 2, 1 that leaves 3 stages in the ring; 1
// whenever K is not a whole number of k-blocks.
int skinny_kgroup(int np, int bm, long long K, int kbe, int kg_req);
// Rows of B per skinny tile chosen automatically for n columns of D and np
// padded tokens.
int skinny_tile_rows(long long n, int np, int max_grid);
// k-parts per tile of the skinny kernel's automatic partition for n columns
// of D (tiles of skinny_tile_rows rows), or 0 where it is stream-K.
int skinny_parts(long long n, int np, int max_grid);

}  // namespace gtn
