// SGMV shrink / expand on the tcgen05 tensor cores: the prefill form of the
// multi-LoRA delta (handbook page "多 LoRA 服务：分段矩阵乘与适配器调度", section
// "不合并权重，批量计算": tokens are stably grouped into same-adapter segments
// and each segment is one small GEMM; page "vLLM 源码完全拆解(十八): 多 LoRA
// 服务", section "两个低秩 GEMM:shrink、expand 与 fp32 中转缓冲").
//
// Work is cut into 128-row tiles of the segments of a work list (the metadata
// kernel's cumulative tile counts). Both kernels are persistent (one CTA per
// SM) and warp-specialised around mbarrier pipelines:
//
// * shrink: item = (tile, split of d_in). Producer warps gather the tile's x
//   rows with 16-byte cp.async into the 128-byte-swizzled K-major operand
//   layout; one of them loads each slice's block of A (64 rows of d_in by
//   r_max) with TMA as a swizzled MN-major operand. One thread issues
//   tcgen05.mma (M = 128, N = r_max per slice, K = 16) into a TMEM
//   accumulator; epilogue warps read it back (tcgen05.ld) and store
//   unscaled fp32 partial rows to the workspace. The number of d_in splits
//   follows the tile count so that every SM gets work (split-K).
// * expand: item = (tile, slice, 128 columns for bf16 y, 64 for fp32 y). The
//   tile's rank-r rows u (scale * the split partials summed in split order,
//   or the caller's buffer) are split into bf16 hi + lo parts and stored once
//   per (tile, slice) as the K-major A operand, so the product keeps fp32
//   accuracy; B blocks come by TMA; y rows come in and go out with per-row
//   bulk copies through shared memory, and the epilogue adds the accumulator
//   (u_hi B + u_lo B) to them in place.
// * reduce: the split path's partials -> buffer rows, with the expand's
//   arithmetic, so split and fused SGMV paths agree bitwise.
//
// Every wait on a barrier is bounded: one that runs out records an error in
// the work-list header (reported by lora_query_status) and the CTA winds
// down without touching memory it does not own.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>

#include "common.cuh"

namespace ra {
namespace {

constexpr int kTileM = LORA_SGMV_TILE_M;  // rows per tile (and MMA M)
constexpr int kKB = 64;                   // d_in elements per shrink K block (one 128-byte swizzle row)
constexpr int kSmemMax = 227 * 1024;
constexpr int kAlignSlack = 1024;         // dynamic smem is re-aligned to 1024 bytes
constexpr int kUKRegion = kTileM * 128;   // bytes of one 64-wide K region of a 128-row operand
constexpr uint64_t kWaitNs = 200000000ull;  // a pipeline wait longer than 200 ms means a fault

// Error bits in the work-list header (word WorkLists::kErrWord).
constexpr int kErrShrink = 1;
constexpr int kErrExpand = 2;
constexpr int kErrProbe = 4;  // lora_probe_bounded_wait

// Shared-memory descriptor layouts.
constexpr uint32_t kSw128 = 2, kSw64 = 4, kSw32 = 6;

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of the given parity. Gives up after limit_ns (by
// default kWaitNs): records `code` in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, int *err, int code,
                                          uint64_t limit_ns = kWaitNs) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try(b, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(err, code);
      return false;
    }
  }
}
// The same, with one verdict for the whole warp (every lane must call it).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *b, uint32_t parity, int *err, int code) {
  return __all_sync(0xffffffffu, mbar_wait(b, parity, err, code)) != 0;
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Order this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
// 16-byte cp.async that writes zeros when !valid (nothing is read then).
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               ::"r"(smem_addr(dst)), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

// TMEM: allocation by one whole warp; the address lands in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_addr(slot)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// MMAs are issued by one elected lane of a converged warp, the way the
// instruction wants its operands (warp-uniform values). A whole 64-deep K
// block (four 16-deep steps) goes out from one asm block: its descriptors are
// formed once and advanced in place, A by a_step and B by b_step (16-byte
// units), so no other instruction sits between the MMAs and the tensor pipe
// stays fed. Timed on this part: back-to-back issue like this keeps an
// M=128 MMA at its pipe rate; with the descriptors rebuilt between MMAs by a
// single divergent lane, issue alone took several times the MMA itself.
// The first MMA accumulates when `acc` is non-zero; the others always do.
// Every lane of the warp must call these.
template <int kSteps>
__device__ __forceinline__ void mma_run(uint32_t d, uint64_t ad, uint64_t bd, uint64_t a_step, uint64_t b_step,
                                        uint32_t idesc, uint32_t acc) {
  static_assert(kSteps == 1 || kSteps == 2 || kSteps == 4, "1, 2 or 4 steps");
  if constexpr (kSteps == 1) {
    asm volatile(
        "{\n\t.reg .pred q, e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 q, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}"
        ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(acc), "l"(a_step), "l"(b_step)
        : "memory");
  } else if constexpr (kSteps == 2) {
    asm volatile(
        "{\n\t.reg .pred q, e, t;\n\t.reg .b32 r;\n\t.reg .b64 a1, b1;\n\t"
        "elect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 q, %4, 0;\n\tsetp.eq.b32 t, %3, %3;\n\t"
        "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t}"
        ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(acc), "l"(a_step), "l"(b_step)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred q, e, t;\n\t.reg .b32 r;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "elect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 q, %4, 0;\n\tsetp.eq.b32 t, %3, %3;\n\t"
        "add.s64 a1, %1, %5;\n\tadd.s64 a2, a1, %5;\n\tadd.s64 a3, a2, %5;\n\t"
        "add.s64 b1, %2, %6;\n\tadd.s64 b2, b1, %6;\n\tadd.s64 b3, b2, %6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}"
        ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(acc), "l"(a_step), "l"(b_step)
        : "memory");
  }
}
// 1, 2 or 4 steps chosen at run time (a warp-uniform value).
__device__ __forceinline__ void mma_steps(int steps, uint32_t d, uint64_t ad, uint64_t bd, uint64_t a_step,
                                          uint64_t b_step, uint32_t idesc, uint32_t acc) {
  if (steps >= 4) mma_run<4>(d, ad, bd, a_step, b_step, idesc, acc);
  else if (steps == 2) mma_run<2>(d, ad, bd, a_step, b_step, idesc, acc);
  else mma_run<1>(d, ad, bd, a_step, b_step, idesc, acc);
}
// D[tmem] (+)= A[smem] * B[smem] with bf16 operands and an fp32 accumulator
// is what each MMA computes. tcgen05.commit, below, gives the barrier one
// arrival once every MMA the committing lane issued so far is complete; it is
// sent from the elected lane, the one that issued the MMAs.
__device__ __forceinline__ void mma_commit_elect(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      ::"r"(smem_addr(bar)) : "memory");
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 accumulator columns, without waiting (see tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (start, leading / stride byte offsets, swizzle).
// For the swizzled MN-major operands here the leading offset is the distance
// between blocks along N and the stride offset the distance between groups of
// 8 rows along K; for the K-major ones the stride offset is the distance
// between groups of 8 rows (the leading offset is unused).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major, B MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Byte offset of 16-byte chunk c of row r in a 128-row, 128-byte-swizzled K-major region.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

// ------------------------------------------------------------------ work items

struct SgList {
  int list;      // int offset of the unit-record list
  int ts;        // int offset of its cumulative tile counts
  int hdr_segs;  // header word: records in the list
  int hdr_tiles; // header word: tiles in the list
};

// The shrink's work: the flattened space of (tile, K block of 64) units,
// U = n_tiles * nb, cut into G contiguous ranges whose sizes differ by at most
// one unit (one per CTA). A CTA's range covers pieces of one or more tiles;
// each piece leaves an unscaled partial at (CTA, piece index in the CTA), and
// a tile's rank-r rows are the sum of its pieces in CTA order.
// At most kMaxFanIn CTAs share a tile (fewer CTAs work when tiles are few),
// which bounds the partials a u row sums.
constexpr int kMaxFanIn = 4;
struct Split {
  int64_t U;
  int G, nb, maxp;  // G: CTAs that take part; maxp: pieces per CTA the workspace holds
  __host__ __device__ __forceinline__ static Split of(int n_tiles, int grid, int nb, int maxp) {
    const int64_t cap = (int64_t)n_tiles * kMaxFanIn;
    return Split{(int64_t)n_tiles * nb, (int)(cap < grid ? (cap > 0 ? cap : 1) : grid), nb, maxp};
  }
  __host__ __device__ __forceinline__ int64_t u0(int c) const { return c < G ? (int64_t)c * U / G : U; }
  // The CTA whose range holds unit u (0 <= u < U).
  __host__ __device__ __forceinline__ int cta_of(int64_t u) const { return (int)(((u + 1) * G - 1) / U); }
};

struct TileInfo {
  int slot, pos0, rows;
};

// The segment of tile `tile`: the last record whose first tile is <= tile.
__device__ __forceinline__ TileInfo tile_info(const int32_t *w, const SgList &L, int n_list, int tile) {
  const int32_t *ts = w + L.ts;
  int lo = 0, hi = n_list - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int32_t *rec = w + L.list + lo * WorkLists::kRec;
  const int k = tile - ts[lo];
  TileInfo t;
  t.slot = rec[1];
  t.pos0 = rec[3] + k * kTileM;
  t.rows = min(kTileM, rec[2] - k * kTileM);
  return t;
}

struct PieceInfo {
  int slot, pos0, rows, tok0, contiguous;
};
constexpr int kPieceCache = 64;  // pieces per CTA whose info is kept in shared memory

__device__ __forceinline__ PieceInfo piece_info(const int32_t *w, const int32_t *sorted_rows, const SgList &L,
                                                int n_list, int tile) {
  const TileInfo ti = tile_info(w, L, n_list, tile);
  PieceInfo p;
  p.slot = ti.slot;
  p.pos0 = ti.pos0;
  p.rows = ti.rows;
  p.tok0 = sorted_rows[ti.pos0];
  p.contiguous = sorted_rows[ti.pos0 + ti.rows - 1] - p.tok0 == ti.rows - 1;
  return p;
}

struct SgMaps {
  CUtensorMap m[LORA_MAX_SLICES];  // A[s] as {r_max, d_in, slots}, boxes of box_n columns x 64 rows
  CUtensorMap x;                   // x as {d_in, T}, boxes of 64 columns x 128 rows (shrink)
};

// ------------------------------------------------------------------ shrink

struct SgShrinkArgs {
  const __nv_bfloat16 *x;
  int64_t ldx;
  float *part;                // partial rows [item][slice][128][r_max]
  const int32_t *work;
  const int32_t *sorted_rows;
  int *err;
  SgList L;
  int d_in, r_max, n_slices, nb, maxp;  // nb: K blocks of 64; maxp: pieces per CTA
  int box_n;                  // TMA box width of an A block (<= 64 columns)
  uint32_t w_layout;          // its swizzle
  int stages, lag, stage_bytes, w_bytes;
  int acc_cols, n_acc, tmem_cols;
  int behind;                 // launched behind this library's BGMV kernel of the same call (see sg_enter)
  int x_div;                  // LoRA row i reads x row i / x_div (> 1: x rows are gathered, never tiled)
};

constexpr int kShrinkProducers = 128;  // warps 0-3
constexpr int kShrinkThreads = 288;    // + epilogue warps 4-7 + MMA warp 8

// Entry and exit of an SGMV kernel. Launched behind this library's BGMV
// kernel of the same call (`behind`), it starts work at once: everything
// older than that kernel is complete when it starts (the BGMV kernel releases
// its successor only after its own wait), the two families touch disjoint
// rows and workspace parts, and its first CTA waits just before it exits, so
// its completion still implies the BGMV kernel's; the other CTAs leave as soon
// as their work is done, handing their SM to the BGMV kernel. Otherwise it
// waits first.
__device__ __forceinline__ void sg_enter(int behind) {
  if (!behind) pdl_wait();
  pdl_trigger();
}
__device__ __forceinline__ void sg_exit(int behind) {
  if (behind && blockIdx.x == 0) pdl_wait();
}

__global__ void __launch_bounds__(kShrinkThreads, 1)
    sgmv_shrink_kernel(const __grid_constant__ SgMaps maps, const SgShrinkArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + a.stages * a.stage_bytes);
  uint64_t *empty = full + a.stages;
  uint64_t *accf = empty + a.stages;
  uint64_t *acce = accf + 2;
  uint64_t *fin = acce + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(fin + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], kShrinkProducers + 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 128);
    }
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  sg_enter(a.behind);
  if (warp == 8) tmem_alloc(tslot, (uint32_t)a.tmem_cols);
  const int n_tiles = a.work[a.L.hdr_tiles];
  const int n_list = a.work[a.L.hdr_segs];
  const Split sp = Split::of(n_tiles, (int)gridDim.x, a.nb, a.maxp);
  const int64_t u0 = sp.u0(blockIdx.x), u1 = sp.u0(blockIdx.x + 1);
  const int t_first = (int)(u0 / a.nb);
  int n_pieces = u1 > u0 ? (int)((u1 - 1) / a.nb) - t_first + 1 : 0;
  if (n_pieces > a.maxp) {  // cannot happen with the host's bound; refuse rather than overrun
    if (tid == 0) atomicOr(a.err, kErrShrink);
    n_pieces = 0;
  }
  // The segment, rows and contiguity of every piece's tile, resolved once
  // (in parallel) before the pipeline starts.
  PieceInfo *pinfo = reinterpret_cast<PieceInfo *>(tslot + 4);
  if (warp == 4)
    for (int p = lane; p < min(n_pieces, kPieceCache); p += 32) pinfo[p] = piece_info(a.work, a.sorted_rows, a.L, n_list, t_first + p);
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = *tslot;

  if (warp < 4) {
    // ---- producers: x rows by cp.async (swizzled), A blocks by TMA (thread 0)
    int issued = 0;
    const int chunk = tid & 7;
    bool ok = true;
    for (int p = 0; p < n_pieces && ok; ++p) {
      const int tile = t_first + p;
      const PieceInfo pi = p < kPieceCache ? pinfo[p] : piece_info(a.work, a.sorted_rows, a.L, n_list, tile);
      const TileInfo ti{pi.slot, pi.pos0, pi.rows};
      // A tile of consecutive tokens comes by one TMA tile copy per K block,
      // already in the swizzled operand layout; others are gathered.
      const int tok0 = pi.tok0;
      const bool contiguous = pi.contiguous != 0 && a.x_div == 1;
      int tok[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = (tid >> 3) + 16 * i;
        tok[i] = (!contiguous && r < ti.rows) ? a.sorted_rows[ti.pos0 + r] : -1;
        if (a.x_div != 1 && tok[i] >= 0) tok[i] /= a.x_div;  // the x row of this LoRA row
      }
      const int kb0 = (int)(max(u0, (int64_t)tile * a.nb) - (int64_t)tile * a.nb);
      const int kb1 = (int)(min(u1, (int64_t)(tile + 1) * a.nb) - (int64_t)tile * a.nb);
      for (int kb = kb0; kb < kb1; ++kb) {
        const int s = issued % a.stages;
        if (!mbar_wait_warp(&empty[s], ((issued / a.stages) & 1) ^ 1, a.err, kErrShrink)) {
          ok = false;
          break;
        }
        unsigned char *st = sm + s * a.stage_bytes;
        // One thread's tensor copies complete one after another (about half a
        // microsecond each, whatever their size), so a stage's copies go out
        // from separate lanes, and the lanes rotate with the stage over eight
        // groups of 16: the group's first lane posts the stage's bytes, then
        // copies x; the next lanes copy one A box each.
        const int grp = issued & 7;
        if (warp == (grp >> 1)) {
          const int l = lane - (grp & 1) * 16;
          if (l == 0) mbar_arrive_tx(&full[s], (uint32_t)(a.n_slices * a.w_bytes + (contiguous ? kTileM * 128 : 0)));
          __syncwarp();
          const int nbx = (a.r_max + a.box_n - 1) / a.box_n;
          if (l == 0 && contiguous) tma_load_2d(st, &maps.x, kb * kKB, tok0, &full[s]);
          if (l >= 1 && l <= a.n_slices * nbx) {
            const int sl = (l - 1) / nbx, bx = (l - 1) - sl * nbx;
            tma_load_3d(st + kTileM * 128 + sl * a.w_bytes + bx * (kKB * a.box_n * 2), &maps.m[sl], bx * a.box_n,
                        kb * kKB, ti.slot, &full[s]);
          }
        }
        if (!contiguous) {
          const int col = kb * kKB + chunk * 8;
          const bool col_ok = col < a.d_in;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (tid >> 3) + 16 * i;
            const bool v = col_ok && tok[i] >= 0;
            const __nv_bfloat16 *src = v ? a.x + (int64_t)tok[i] * a.ldx + col : a.x;
            cp_async16_zfill(st + swz128(r, chunk), src, v);
          }
        }
        cp_async_commit();
        ++issued;
        if (issued > a.lag) {
          cp_async_wait_upto(a.lag);
          fence_async_smem();
          mbar_arrive(&full[(issued - 1 - a.lag) % a.stages]);
        }
      }
    }
    cp_async_wait_upto(0);
    fence_async_smem();
    for (int j = issued - a.lag < 0 ? 0 : issued - a.lag; j < issued; ++j) mbar_arrive(&full[j % a.stages]);
  } else if (warp < 8) {
    // ---- epilogue: accumulator -> unscaled partial rows (thread = row)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int nitem = 0;
    for (int p = 0; p < n_pieces; ++p) {
      const int acc = nitem % a.n_acc;
      if (!mbar_wait_warp(&accf[acc], (nitem / a.n_acc) & 1, a.err, kErrShrink)) break;
      tc_after_sync();
      const uint32_t t0 = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * a.acc_cols);
      for (int sl = 0; sl < a.n_slices; ++sl) {
        float *dst = a.part + ((((int64_t)blockIdx.x * a.maxp + p) * a.n_slices + sl) * kTileM + row) * a.r_max;
        for (int c = 0; c < a.r_max; c += 16) {
          float v[16];
          tmem_ld16(t0 + (uint32_t)(sl * a.r_max + c), v);
          float4 *d4 = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
          for (int j = 0; j < 4; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      tc_before_sync();
      mbar_arrive(&acce[acc]);
      ++nitem;
    }
  } else {
    // ---- MMA issuer: the whole warp walks the pipeline, one elected lane issues.
    // The slices' A blocks sit side by side at one stride, so up to 256 columns
    // (gsl slices) go into one MMA.
    const int gsl = min(a.n_slices, max(1, 256 / a.r_max));
    const int n_groups = (a.n_slices + gsl - 1) / gsl;
    const uint32_t sbo_w = 8u * a.box_n * 2, lbo_w = (uint32_t)kKB * a.box_n * 2;
    const uint64_t b_step = (2u * sbo_w) >> 4;  // 16 K rows of the MN-major block
    const uint32_t id_full = idesc_bf16(kTileM, gsl * a.r_max);
    const uint32_t id_last = idesc_bf16(kTileM, (a.n_slices - (n_groups - 1) * gsl) * a.r_max);
    int consumed = 0, nitem = 0;
    bool ok = true;
    for (int p = 0; p < n_pieces && ok; ++p) {
      const int tile = t_first + p;
      const int kb0 = (int)(max(u0, (int64_t)tile * a.nb) - (int64_t)tile * a.nb);
      const int kb1 = (int)(min(u1, (int64_t)(tile + 1) * a.nb) - (int64_t)tile * a.nb);
      const int acc = nitem % a.n_acc;
      if (!mbar_wait_warp(&acce[acc], ((nitem / a.n_acc) & 1) ^ 1, a.err, kErrShrink)) break;
      tc_after_sync();
      const uint32_t d0 = tmem + (uint32_t)(acc * a.acc_cols);
      for (int kb = kb0; kb < kb1; ++kb) {
        const int s = consumed % a.stages;
        if (!mbar_wait_warp(&full[s], (consumed / a.stages) & 1, a.err, kErrShrink)) {
          ok = false;
          break;
        }
        tc_after_sync();
        const uint32_t xs = smem_addr(sm + s * a.stage_bytes);
        const uint64_t ad = smem_desc(xs, 16, 1024, kSw128);
        for (int g = 0; g < n_groups; ++g) {
          const uint64_t bd = smem_desc(xs + kTileM * 128 + g * gsl * a.w_bytes, lbo_w, sbo_w, a.w_layout);
          mma_run<kKB / 16>(d0 + (uint32_t)(g * gsl * a.r_max), ad, bd, 2, b_step, g + 1 < n_groups ? id_full : id_last,
                            kb > kb0 ? 1u : 0u);
        }
        mma_commit_elect(&empty[s]);
        ++consumed;
      }
      if (!ok) break;
      mma_commit_elect(&accf[acc]);
      ++nitem;
    }
    mma_commit_elect(fin);
    mbar_wait_warp(fin, 0, a.err, kErrShrink);  // every MMA is done before TMEM is freed
  }
  tc_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc_after_sync();
    tmem_free(tmem, (uint32_t)a.tmem_cols);
  }
  sg_exit(a.behind);
}

// ------------------------------------------------------------------ u rows (expand and reduce)

struct URowArgs {
  const float *src;  // partials [CTA][piece][slice][128][r_max], or buf [n_s, T, r_max]
  int parts;
  Split sp;          // the shrink's partition (parts only)
  int n_slices, r_max, T;
};

// u[k] for 16 consecutive k (k0 multiple of 16) of one row: scale * the
// tile's pieces summed in CTA order (masked to the slot's rank), or the
// buffer. The loads of FB pieces are issued together, then summed in order,
// so a row waits for one round trip per FB pieces (the reduce kernel takes
// FB = 4; the expand's loader warps keep FB = 1, which leaves the registers
// its epilogue warps need).
template <int FB>
__device__ __forceinline__ void u_row16(const URowArgs &u, int tile, int slice, int row, int tok, int k0, int r_a,
                                        float scale, float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = 0.f;
  if (k0 >= r_a) return;
  if (u.parts) {
    const int c0 = u.sp.cta_of((int64_t)tile * u.sp.nb), c1 = u.sp.cta_of((int64_t)(tile + 1) * u.sp.nb - 1);
    if constexpr (FB == 1) {
      for (int c = c0; c <= c1; ++c) {
        const int64_t cu0 = u.sp.u0(c);
        if (u.sp.u0(c + 1) == cu0) continue;  // fewer units than CTAs: this CTA has none
        const int j = tile - (int)(cu0 / u.sp.nb);
        const float4 *p = reinterpret_cast<const float4 *>(
            u.src + ((((int64_t)c * u.sp.maxp + j) * u.n_slices + slice) * kTileM + row) * u.r_max + k0);
        float4 q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = p[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] += q[i].x;
          v[4 * i + 1] += q[i].y;
          v[4 * i + 2] += q[i].z;
          v[4 * i + 3] += q[i].w;
        }
      }
    } else {
      for (int cb = c0; cb <= c1; cb += FB) {
        float4 q[FB][4];
        bool have[FB];
#pragma unroll
        for (int b = 0; b < FB; ++b) {
          const int c = cb + b;
          const int64_t cu0 = c <= c1 ? u.sp.u0(c) : 0;
          have[b] = c <= c1 && u.sp.u0(c + 1) != cu0;  // fewer units than CTAs: a CTA may have none
          if (have[b]) {
            const int j = tile - (int)(cu0 / u.sp.nb);
            const float4 *p = reinterpret_cast<const float4 *>(
                u.src + ((((int64_t)c * u.sp.maxp + j) * u.n_slices + slice) * kTileM + row) * u.r_max + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) q[b][i] = p[i];
          }
        }
#pragma unroll
        for (int b = 0; b < FB; ++b) {
          if (!have[b]) continue;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[4 * i] += q[b][i].x;
            v[4 * i + 1] += q[b][i].y;
            v[4 * i + 2] += q[b][i].z;
            v[4 * i + 3] += q[b][i].w;
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] *= scale;
  } else {
    const float4 *p = reinterpret_cast<const float4 *>(u.src + ((int64_t)slice * u.T + tok) * u.r_max + k0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = p[i];
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (k0 + j >= r_a) v[j] = 0.f;
}

// ------------------------------------------------------------------ reduce (split path)

struct SgReduceArgs {
  URowArgs u;
  float *buf;
  const int32_t *work;
  const int32_t *sorted_rows;
  const int32_t *slot_rank;
  const float *slot_scale;
  int *err;
  SgList L;
  int shrink_grid, nb, maxp;
};

// Grid-stride over (tile, slice); thread = row.
__global__ void __launch_bounds__(kTileM) sgmv_reduce_kernel(const SgReduceArgs a) {
  pdl_wait();
  pdl_trigger();
  const int n_tiles = a.work[a.L.hdr_tiles];
  const int n_list = a.work[a.L.hdr_segs];
  URowArgs u = a.u;
  u.sp = Split::of(n_tiles, a.shrink_grid, a.nb, a.maxp);
  const int row = threadIdx.x;
  for (int p = blockIdx.x; p < n_tiles * u.n_slices; p += gridDim.x) {
    const int tile = p / u.n_slices, slice = p - tile * u.n_slices;
    const TileInfo ti = tile_info(a.work, a.L, n_list, tile);
    if (row >= ti.rows) continue;
    const int tok = a.sorted_rows[ti.pos0 + row];
    const int r_a = min(max(a.slot_rank[ti.slot], 0), u.r_max);
    const float scale = a.slot_scale[ti.slot];
    float *dst = a.buf + ((int64_t)slice * u.T + tok) * u.r_max;
    for (int k0 = 0; k0 < u.r_max; k0 += 16) {
      float v[16];
      u_row16<4>(u, tile, slice, row, tok, k0, r_a, scale, v);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<float4 *>(dst + k0)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

// ------------------------------------------------------------------ expand

struct SgExpandArgs {
  URowArgs u;
  void *y;
  int64_t ldy;
  const int32_t *work;
  const int32_t *sorted_rows;
  const int32_t *slot_rank;
  const float *slot_scale;
  int *err;
  SgList L;
  int shrink_grid, nb, maxp;
  int out_sizes[LORA_MAX_SLICES];
  int out_off[LORA_MAX_SLICES];
  int nb_start[LORA_MAX_SLICES + 1];  // column blocks per slice (cumulative)
  int nk;                             // 64-wide K regions of the u operand (1 or 2)
  int b_stages, y_stages, b_bytes;
  int behind;                         // launched behind this library's BGMV kernel of the same call
};

struct SgExpandMaps {
  CUtensorMap b[LORA_MAX_SLICES];  // B[s] as {out_s, r_max, slots}, boxes of 64 columns x r_max rows
  CUtensorMap y;                   // y as {sum(out_sizes), T}, boxes of 128 bytes x 128 rows (loads)
  CUtensorMap ys;                  // the same y, boxes of 128 bytes x 32 rows (an epilogue warp's store)
};

constexpr int kEpiWarps = 8;  // epilogue warps, a multiple of 4 (one group per TMEM lane quadrant); 8 measured best
// Accumulators in the expand's ring: the MMA warp runs up to kExpandAcc - 1
// items ahead of the epilogue, so neither waits on the other's latency (with
// two, an item took the MMA time plus the epilogue's hand-off). 4 x 128
// columns fill the 512 TMEM columns for a bf16 y.
constexpr int kExpandAcc = 4;
constexpr int kExpandThreads = 32 * (kEpiWarps + 6);  // + loaders (u rows, gathered y rows) x4, producer, MMA
constexpr int kYHalf = kTileM * 128;  // one half (128 bytes per row) of a staged y tile
constexpr int kYStage = 2 * kYHalf;   // a staged y tile: 128 rows x 256 bytes

template <typename TY> struct YCols { static constexpr int kN = 256 / (int)sizeof(TY); };  // 256 bytes per row

struct ExpandItem {
  int tile, slice, n0, ncols, group;
};

__device__ __forceinline__ ExpandItem expand_item(const SgExpandArgs &a, int64_t it, int nbt, int kN, int n_slices) {
  ExpandItem e;
  e.tile = (int)(it / nbt);
  const int j = (int)(it - (int64_t)e.tile * nbt);
  int s = 0;
  while (s + 1 < n_slices && j >= a.nb_start[s + 1]) ++s;
  e.slice = s;
  e.n0 = (j - a.nb_start[s]) * kN;
  e.ncols = min(kN, a.out_sizes[s] - e.n0);
  e.group = e.tile * n_slices + s;
  return e;
}

// Offset of 16-byte chunk g (0..15) of row r in a staged y tile: two halves
// of 128-byte rows in the 128-byte swizzle that the tile copy writes.
__device__ __forceinline__ uint32_t ychunk(int r, int g) {
  return (uint32_t)((g >> 3) * kYHalf + r * 128 + (((g & 7) ^ (r & 7)) << 4));
}

// A tile and whether its rows are one run of consecutive tokens (then its y
// rows arrive as two TMA tile copies; otherwise loader warps gather them).
struct TileRows {
  int tile = -1;
  TileInfo ti{0, 0, 0};
  int tok0 = 0;
  bool contiguous = false;
  __device__ __forceinline__ bool at(const SgExpandArgs &a, int n_list, int t) {
    if (t == tile) return false;
    ti = tile_info(a.work, a.L, n_list, t);
    tok0 = a.sorted_rows[ti.pos0];
    contiguous = a.sorted_rows[ti.pos0 + ti.rows - 1] - tok0 == ti.rows - 1;
    tile = t;
    return true;
  }
};

// One elected lane stores a box of the staged tile with a TMA tile copy and
// closes it as a bulk group; the same lane later waits for the group's
// shared-memory reads (the slot may then be refilled) or for its completion.
__device__ __forceinline__ void tma_store_2d_elect(const CUtensorMap *map, const void *src, int c0, int c1) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n\t"
      "@e cp.async.bulk.commit_group;\n\t}"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(c0), "r"(c1)
      : "memory");
}
template <int kPending>
__device__ __forceinline__ void bulk_wait_read_elect() {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.wait_group.read %0;\n\t}" ::"n"(kPending) : "memory");
}
__device__ __forceinline__ void bulk_wait_all_elect() {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.wait_group 0;\n\t}" ::: "memory");
}

// The barrier receives this thread's arrival once its earlier cp.async copies are complete.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <typename TY>
__global__ void __launch_bounds__(kExpandThreads, 1)
    sgmv_expand_kernel(const __grid_constant__ SgExpandMaps maps, const SgExpandArgs a) {
  constexpr int kN = YCols<TY>::kN;           // columns per item (256 bytes of a y row)
  constexpr int kVec = 16 / (int)sizeof(TY);  // y elements per 16-byte chunk
  constexpr int kHalf = kN / 2;               // columns per 128-byte staged half
  constexpr int kParts = kEpiWarps / 4;       // epilogue warps per TMEM lane quadrant
  constexpr int kPartCols = kN / kParts;      // accumulator columns per epilogue warp
  constexpr int kPartChunks = 16 / kParts;    // 16-byte chunks per row in a part
  constexpr int kRowsPerInst = 32 / kPartChunks;
  constexpr int kStoreInsts = 32 / kRowsPerInst;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const int r_max = a.u.r_max, n_slices = a.u.n_slices;
  unsigned char *sU = sm;                                  // hi: nk regions, then lo: nk regions
  unsigned char *sB = sU + 2 * a.nk * kUKRegion;
  unsigned char *sY = sB + a.b_stages * a.b_bytes;
  uint64_t *bfull = reinterpret_cast<uint64_t *>(sY + a.y_stages * kYStage);
  uint64_t *bempty = bfull + a.b_stages;
  uint64_t *yfull = bempty + a.b_stages;
  uint64_t *yempty = yfull + a.y_stages;
  uint64_t *accf = yempty + a.y_stages;
  uint64_t *acce = accf + kExpandAcc;
  uint64_t *ufull = acce + kExpandAcc;
  uint64_t *uempty = ufull + 1;
  uint64_t *fin = uempty + 1;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(fin + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < a.b_stages; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < a.y_stages; ++s) {
      mbar_init(&yfull[s], 1 + 128);  // the producer + every loader thread
      mbar_init(&yempty[s], 32 * kEpiWarps);
    }
    for (int i = 0; i < kExpandAcc; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 32 * kEpiWarps);
    }
    mbar_init(ufull, 128);
    mbar_init(uempty, 1);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  sg_enter(a.behind);
  constexpr uint32_t kTmemCols = kExpandAcc * kN;
  static_assert(kTmemCols <= 512, "accumulators exceed tensor memory");
  if (warp == kEpiWarps + 5) tmem_alloc(tslot, kTmemCols);
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = *tslot;
  const int n_tiles = a.work[a.L.hdr_tiles];
  const int n_list = a.work[a.L.hdr_segs];
  const int nbt = a.nb_start[n_slices];
  const int64_t n_items = (int64_t)n_tiles * nbt;
  int64_t it0, it1;
  if ((int64_t)n_tiles * kMaxFanIn <= gridDim.x) {
    // Few tiles: each tile gets its own CTAs (as many per tile as the grid
    // allows, within one) and a CTA's items never cross into the next tile,
    // so no CTA forms the u rows of two tiles one after the other.
    const int t = (int)((int64_t)blockIdx.x * n_tiles / gridDim.x);  // tile t's CTAs: [ceil(t G / n), ceil((t + 1) G / n))
    const int cb = (int)(((int64_t)t * gridDim.x + n_tiles - 1) / n_tiles);
    const int ce = (int)(((int64_t)(t + 1) * gridDim.x + n_tiles - 1) / n_tiles);
    const int k = (int)blockIdx.x - cb, nk = ce - cb;
    it0 = (int64_t)t * nbt + (int64_t)nbt * k / nk;
    it1 = (int64_t)t * nbt + (int64_t)nbt * (k + 1) / nk;
  } else {
    it0 = n_items * blockIdx.x / gridDim.x;
    it1 = n_items * (blockIdx.x + 1) / gridDim.x;
  }
  TY *y = static_cast<TY *>(a.y);

  if (warp < kEpiWarps) {
    // ---- epilogue. Warp w adds accumulator lanes 32 (w % 4), column part
    // w / 4 (kPartCols columns), into the staged rows (thread = row), then
    // stores that part of its 32 rows with coalesced 16-byte stores.
    const int q = warp & 3, part = warp >> 2;
    const int row = q * 32 + lane;
    const int g0 = part * kPartChunks;  // first 16-byte chunk of this part
    int cur_tile = -1, tok = -1, nitem = 0;
    int tok0 = 0;                 // first token of the tile when its rows are one run of tokens
    bool whole_rows = false;      // ... and this warp's 32 rows are all tokens of it
    int pend = -1;                // ring slot whose bulk store may still be reading it
    int stok[kStoreInsts];
#pragma unroll
    for (int i = 0; i < kStoreInsts; ++i) stok[i] = -1;
    for (int64_t it = it0; it < it1; ++it) {
      const ExpandItem e = expand_item(a, it, nbt, kN, n_slices);
      if (e.tile != cur_tile) {
        const TileInfo ti = tile_info(a.work, a.L, n_list, e.tile);
        tok = row < ti.rows ? a.sorted_rows[ti.pos0 + row] : -1;
#pragma unroll
        for (int i = 0; i < kStoreInsts; ++i) {
          const int r = 32 * q + kRowsPerInst * i + lane / kPartChunks;
          stok[i] = r < ti.rows ? a.sorted_rows[ti.pos0 + r] : -1;
        }
        tok0 = a.sorted_rows[ti.pos0];
        whole_rows = 32 * q + 32 <= ti.rows && a.sorted_rows[ti.pos0 + ti.rows - 1] - tok0 == ti.rows - 1;
        cur_tile = e.tile;
      }
      const int acc = nitem % kExpandAcc, ys = nitem % a.y_stages;
      const uint32_t par = (nitem / a.y_stages) & 1;
      if (!mbar_wait_warp(&accf[acc], (nitem / kExpandAcc) & 1, a.err, kErrExpand)) break;
      tc_after_sync();
      float v[kPartCols];
      const uint32_t t0 = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kN + part * kPartCols);
      if constexpr (kPartCols >= 32) {
#pragma unroll
        for (int c = 0; c < kPartCols; c += 32) tmem_ld32_async(t0 + (uint32_t)c, v + c);
        tmem_wait_ld();
      } else {
        float v16[16];
        tmem_ld16(t0, v16);
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = v16[c];
      }
      tc_before_sync();
      mbar_arrive(&acce[acc]);
      if (!mbar_wait_warp(&yfull[ys], par, a.err, kErrExpand)) break;
      unsigned char *st = sY + ys * kYStage;
      if (tok >= 0) {  // this row's part: all its chunks in flight at once
        uint4 w[kPartChunks];
#pragma unroll
        for (int g = 0; g < kPartChunks; ++g) w[g] = *reinterpret_cast<const uint4 *>(st + ychunk(row, g0 + g));
#pragma unroll
        for (int g = 0; g < kPartChunks; ++g) {
          if constexpr (sizeof(TY) == 2) {
            uint32_t *u32 = reinterpret_cast<uint32_t *>(&w[g]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = make_float2(__uint_as_float(u32[j] << 16), __uint_as_float(u32[j] & 0xffff0000u));
              const float2 sum = __fadd2_rn(f, make_float2(v[g * 8 + 2 * j], v[g * 8 + 2 * j + 1]));
              const __nv_bfloat162 b = __floats2bfloat162_rn(sum.x, sum.y);
              u32[j] = *reinterpret_cast<const uint32_t *>(&b);
            }
          } else {
            float *f = reinterpret_cast<float *>(&w[g]);
            const float2 lo = __fadd2_rn(make_float2(f[0], f[1]), make_float2(v[g * 4], v[g * 4 + 1]));
            const float2 hi = __fadd2_rn(make_float2(f[2], f[3]), make_float2(v[g * 4 + 2], v[g * 4 + 3]));
            f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
          }
        }
#pragma unroll
        for (int g = 0; g < kPartChunks; ++g) *reinterpret_cast<uint4 *>(st + ychunk(row, g0 + g)) = w[g];
      }
      // Store this warp's part of its 32 rows. When the rows are 32
      // consecutive tokens and the part lies inside the slice, one bulk tile
      // store sends it straight from the staged (swizzled) tile; otherwise
      // lanes along the row, kRowsPerInst rows per instruction, and columns
      // past the slice stay unstored.
      const bool bulk = whole_rows && part * kPartCols + kPartCols <= e.ncols;
      if (bulk) {
        fence_async_smem();  // this lane's staged writes, before the copy reads them
        __syncwarp();
        tma_store_2d_elect(&maps.ys, st + part * kYHalf + q * 32 * 128, a.out_off[e.slice] + e.n0 + part * kPartCols,
                           tok0 + 32 * q);
      } else {
        __syncwarp();
        const int gl = lane % kPartChunks;
        if ((g0 + gl) * kVec < e.ncols) {
          TY *ybase = y + a.out_off[e.slice] + e.n0 + (g0 + gl) * kVec;
          uint4 w[kStoreInsts];
#pragma unroll
          for (int i = 0; i < kStoreInsts; ++i)
            w[i] = *reinterpret_cast<const uint4 *>(st + ychunk(32 * q + kRowsPerInst * i + lane / kPartChunks, g0 + gl));
#pragma unroll
          for (int i = 0; i < kStoreInsts; ++i)
            if (stok[i] >= 0) *reinterpret_cast<uint4 *>(ybase + (int64_t)stok[i] * a.ldy) = w[i];
        }
      }
      // A slot goes back to the loaders once nothing reads it: at once after
      // lane stores, one item later after a bulk store (its reads are done
      // when at most the newest group is still pending).
      if (pend >= 0) {
        if (bulk) bulk_wait_read_elect<1>();
        else bulk_wait_read_elect<0>();
        __syncwarp();
        mbar_arrive(&yempty[pend]);
        pend = -1;
      }
      if (bulk) pend = ys;
      else mbar_arrive(&yempty[ys]);
      ++nitem;
    }
    if (pend >= 0) {
      bulk_wait_read_elect<0>();
      __syncwarp();
      mbar_arrive(&yempty[pend]);
    }
    bulk_wait_all_elect();  // every bulk store has landed before the CTA exits
  } else if (warp < kEpiWarps + 4) {
    // ---- loaders: the u rows of each (tile, slice) (thread = row), and the
    // y rows of tiles that are not one run of tokens (16-byte cp.async,
    // lanes along a row)
    const int lt = tid - 32 * kEpiWarps;
    const int wb = lt >> 5;
    URowArgs u = a.u;
    u.sp = Split::of(n_tiles, a.shrink_grid, a.nb, a.maxp);
    int cur_group = -1, g = 0, nitem = 0;
    TileRows tr;
    int ltok[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ltok[i] = -1;
    for (int64_t it = it0; it < it1; ++it) {
      const ExpandItem e = expand_item(a, it, nbt, kN, n_slices);
      if (tr.at(a, n_list, e.tile)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 8 * i + 2 * wb + (lane >> 4);
          ltok[i] = r < tr.ti.rows ? a.sorted_rows[tr.ti.pos0 + r] : -1;
        }
      }
      if (e.group != cur_group) {
        cur_group = e.group;
        const int tok = lt < tr.ti.rows ? a.sorted_rows[tr.ti.pos0 + lt] : -1;
        const int r_a = tok >= 0 ? min(max(a.slot_rank[tr.ti.slot], 0), r_max) : 0;
        const float scale = a.slot_scale[tr.ti.slot];
        if (!mbar_wait_warp(uempty, (g & 1) ^ 1, a.err, kErrExpand)) break;
        for (int k0 = 0; k0 < r_max; k0 += 16) {
          float v[16];
          u_row16<1>(u, e.tile, e.slice, lt, tok, k0, r_a, scale, v);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {  // two 16-byte chunks of 8 k values
            uint4 hi, lo;
            __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&hi);
            __nv_bfloat162 *l2 = reinterpret_cast<__nv_bfloat162 *>(&lo);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __nv_bfloat162 hh = __floats2bfloat162_rn(v[8 * hc + 2 * j], v[8 * hc + 2 * j + 1]);
              const float2 hf = __bfloat1622float2(hh);
              h2[j] = hh;
              l2[j] = __floats2bfloat162_rn(v[8 * hc + 2 * j] - hf.x, v[8 * hc + 2 * j + 1] - hf.y);
            }
            const int c = k0 / 8 + hc;
            const uint32_t off = (uint32_t)((c >> 3) * kUKRegion) + swz128(lt, c & 7);
            *reinterpret_cast<uint4 *>(sU + off) = hi;
            *reinterpret_cast<uint4 *>(sU + a.nk * kUKRegion + off) = lo;
          }
        }
        fence_async_smem();
        mbar_arrive(ufull);
        ++g;
      }
      const int ys = nitem % a.y_stages;
      if (!mbar_wait_warp(&yempty[ys], ((nitem / a.y_stages) & 1) ^ 1, a.err, kErrExpand)) break;
      if (!tr.contiguous) {
        unsigned char *st = sY + ys * kYStage;
        const int gg = lane & 15;
        const bool col_ok = gg * kVec < e.ncols;
        const TY *src0 = y + a.out_off[e.slice] + e.n0 + gg * kVec;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 8 * i + 2 * wb + (lane >> 4);
          if (col_ok && ltok[i] >= 0) cp_async16(st + ychunk(r, gg), src0 + (int64_t)ltok[i] * a.ldy);
        }
      }
      cp_async_arrive(&yfull[ys]);
      ++nitem;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kEpiWarps + 4) {
    // ---- producer: B blocks, and y rows of contiguous tiles, by TMA
    TileRows tr;
    int nitem = 0;
    for (int64_t it = it0; it < it1; ++it) {
      const ExpandItem e = expand_item(a, it, nbt, kN, n_slices);
      tr.at(a, n_list, e.tile);
      const int bs = nitem % a.b_stages, ys = nitem % a.y_stages;
      if (!mbar_wait_warp(&bempty[bs], ((nitem / a.b_stages) & 1) ^ 1, a.err, kErrExpand)) break;
      if (lane == 0) {
        const int nbox = (e.ncols + 63) / 64;  // boxes entirely past the slice are not loaded
        mbar_arrive_tx(&bfull[bs], (uint32_t)(nbox * r_max * 128));
        for (int bx = 0; bx < nbox; ++bx)
          tma_load_3d(sB + bs * a.b_bytes + bx * r_max * 128, &maps.b[e.slice], e.n0 + 64 * bx, 0, tr.ti.slot,
                      &bfull[bs]);
      }
      if (!mbar_wait_warp(&yempty[ys], ((nitem / a.y_stages) & 1) ^ 1, a.err, kErrExpand)) break;
      if (lane == 0) {
        if (tr.contiguous) {
          const int halves = e.ncols > kHalf ? 2 : 1;
          unsigned char *st = sY + ys * kYStage;
          mbar_arrive_tx(&yfull[ys], (uint32_t)(halves * kYHalf));
          for (int hh = 0; hh < halves; ++hh)
            tma_load_2d(st + hh * kYHalf, &maps.y, a.out_off[e.slice] + e.n0 + hh * kHalf, tr.tok0, &yfull[ys]);
        } else {
          mbar_arrive(&yfull[ys]);
        }
      }
      ++nitem;
    }
  } else if (warp == kEpiWarps + 5) {
    // ---- MMA issuer: acc = u_hi B + u_lo B, K = r_max each. The whole warp
    // walks the items, one elected lane issues (a 64-deep K block per run).
    const uint32_t idesc = idesc_bf16(kTileM, kN);
    const uint32_t uhi = smem_addr(sU), ulo = uhi + (uint32_t)(a.nk * kUKRegion);
    const uint32_t lbo_b = (uint32_t)r_max * 128;
    const int steps = min(r_max, 64) / 16;  // 16-deep K steps per 64-deep block (r_max 16, 32: 1, 2)
    int cur_group = -1, g = 0, nitem = 0;
    for (int64_t it = it0; it < it1; ++it) {
      const ExpandItem e = expand_item(a, it, nbt, kN, n_slices);
      if (e.group != cur_group) {
        if (cur_group >= 0) mma_commit_elect(uempty);  // the previous u rows are free once its MMAs finish
        if (!mbar_wait_warp(ufull, g & 1, a.err, kErrExpand)) break;
        ++g;
        cur_group = e.group;
      }
      const int acc = nitem % kExpandAcc, bs = nitem % a.b_stages;
      if (!mbar_wait_warp(&acce[acc], ((nitem / kExpandAcc) & 1) ^ 1, a.err, kErrExpand)) break;
      if (!mbar_wait_warp(&bfull[bs], (nitem / a.b_stages) & 1, a.err, kErrExpand)) break;
      tc_after_sync();
      const uint32_t d = tmem + (uint32_t)(acc * kN);
      const uint32_t bb = smem_addr(sB + bs * a.b_bytes);
      // K block c covers u columns [64c, 64c + 64): its own u region, B rows 64c on.
      for (int c = 0; c < a.nk; ++c) {
        const uint64_t bd = smem_desc(bb + c * 4 * 2048, lbo_b, 1024, kSw128);
        mma_steps(steps, d, smem_desc(uhi + c * kUKRegion, 16, 1024, kSw128), bd, 2, 128, idesc, c > 0 ? 1u : 0u);
      }
      for (int c = 0; c < a.nk; ++c) {
        const uint64_t bd = smem_desc(bb + c * 4 * 2048, lbo_b, 1024, kSw128);
        mma_steps(steps, d, smem_desc(ulo + c * kUKRegion, 16, 1024, kSw128), bd, 2, 128, idesc, 1u);
      }
      mma_commit_elect(&bempty[bs]);
      mma_commit_elect(&accf[acc]);
      ++nitem;
    }
    mma_commit_elect(fin);
    mbar_wait_warp(fin, 0, a.err, kErrExpand);  // every MMA is done before TMEM is freed
  }
  tc_before_sync();
  __syncthreads();
  if (warp == kEpiWarps + 5) {
    tc_after_sync();
    tmem_free(tmem, kTmemCols);
  }
  sg_exit(a.behind);
}

// ------------------------------------------------------------------ host side

int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor map {d0 (contiguous), d1, d2} with a {box0, box1, 1} box.
cudaError_t make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                     uint32_t box1, CUtensorMapSwizzle sw) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D tensor map of a row-major matrix {cols (contiguous), rows} with row
// stride `ld` elements, boxes of box_cols columns (128 bytes) x box_rows rows
// in the 128-byte swizzle.
cudaError_t make_rows_map(CUtensorMap *m, const void *base, bool bf16, uint64_t cols, uint64_t rows, int64_t ld,
                          uint32_t box_cols, uint32_t box_rows = kTileM) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const uint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * es};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                   const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

SgList list_of(const MetaView &mv, ListSel sel) {
  SgList L;
  L.list = WorkLists::list(mv.num_slots, sel);
  if (sel == kListLarge) {
    L.ts = WorkLists::large_tile_start(mv.num_slots);
    L.hdr_segs = 2;
    L.hdr_tiles = 4;
  } else {
    L.ts = WorkLists::all_tile_start(mv.num_slots);
    L.hdr_segs = 0;
    L.hdr_tiles = 3;
  }
  return L;
}

int nb_of(const lora_layer_desc &d) { return (d.d_in + kKB - 1) / kKB; }

// Upper bound on the tiles of any work list for T tokens and S slots.
int64_t tiles_bound(int T, int S) { return (int64_t)T / kTileM + std::min<int64_t>(S - 1, T); }

int shrink_grid() { return sm_count(); }

// Pieces per CTA of the shrink's partition, for any batch of T tokens: a
// range of at most ceil(U / G) units spans at most n_tiles / G + 2 tiles.
int maxp_of(int T, int S, int G) { return (int)(tiles_bound(T, S) / G) + 2; }

// The pipelines' bounded wait on a barrier that nothing will ever arm: one
// thread initialises an mbarrier expecting one arrival and waits for its
// first phase with a limit of limit_ns; no copy or MMA is issued, so when the
// wait gives up (recording kErrProbe) nothing of this kernel is in flight.
__global__ void __launch_bounds__(32) wait_probe_kernel(int *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    (void)mbar_wait(&bar, 0, err, kErrProbe, limit_ns);
  }
}

}  // namespace

bool sgmv_supported() { return encode_fn() != nullptr; }

cudaError_t launch_wait_probe(const MetaView &mv, uint32_t limit_us, cudaStream_t st) {
  int *err = const_cast<int32_t *>(mv.work) + WorkLists::kErrWord;
  return launch_pdl(wait_probe_kernel, dim3(1), dim3(32), 0, st, 1u, err, (uint64_t)limit_us * 1000ull);
}

size_t sgmv_workspace_bytes(const lora_layer_desc &d, int max_tokens) {
  if (max_tokens <= 0) return 0;
  const int G = shrink_grid();
  if (G <= 0) return 0;
  const int64_t pieces = (int64_t)G * maxp_of(max_tokens, d.num_slots, G);
  return (size_t)pieces * d.n_slices * kTileM * d.r_max * sizeof(float);
}

cudaError_t launch_sgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x, int64_t ldx,
                               float *part, cudaStream_t st, bool behind) {
  if (mv.num_tokens <= 0 || mv.num_slots <= 1) return cudaSuccess;
  SgMaps maps;
  memset(&maps, 0, sizeof(maps));
  SgShrinkArgs a{};
  a.box_n = d.r_max < 64 ? d.r_max : 64;
  const CUtensorMapSwizzle sw = a.box_n == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : a.box_n == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  a.w_layout = a.box_n == 64 ? kSw128 : a.box_n == 32 ? kSw64 : kSw32;
  for (int s = 0; s < d.n_slices; ++s) {
    cudaError_t e = make_map(&maps.m[s], d.A[s], (uint64_t)d.r_max, (uint64_t)d.d_in, (uint64_t)d.num_slots,
                             (uint32_t)a.box_n, (uint32_t)kKB, sw);
    if (e != cudaSuccess) return e;
  }
  a.x_div = d.x_row_div > 1 ? d.x_row_div : 1;
  {
    const uint64_t x_rows = ((uint64_t)mv.num_tokens + a.x_div - 1) / a.x_div;
    cudaError_t e = make_rows_map(&maps.x, x, true, (uint64_t)d.d_in, x_rows, ldx, kKB);
    if (e != cudaSuccess) return e;
  }
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.ldx = ldx;
  a.part = part;
  a.behind = behind ? 1 : 0;
  a.work = mv.work;
  a.sorted_rows = mv.sorted_rows;
  a.err = const_cast<int32_t *>(mv.work) + WorkLists::kErrWord;
  a.L = list_of(mv, sel);
  a.d_in = d.d_in;
  a.r_max = d.r_max;
  a.n_slices = d.n_slices;
  a.nb = nb_of(d);
  a.maxp = maxp_of(mv.num_tokens, mv.num_slots, shrink_grid());
  a.w_bytes = kKB * d.r_max * 2;
  a.stage_bytes = kTileM * 128 + d.n_slices * a.w_bytes;
  const int fixed = kAlignSlack + 2048;  // barriers, TMEM address, piece cache
  a.stages = std::min(6, (kSmemMax - fixed) / a.stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidValue;
  a.lag = std::min(2, a.stages - 1);
  a.acc_cols = d.n_slices * d.r_max;
  a.n_acc = 2 * a.acc_cols <= 512 ? 2 : 1;
  int cols = 32;
  while (cols < a.n_acc * a.acc_cols) cols *= 2;
  a.tmem_cols = cols;
  const int smem = fixed + a.stages * a.stage_bytes;
  cudaError_t e = set_max_dynamic_smem((const void *)sgmv_shrink_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sgmv_shrink_kernel, dim3((unsigned)shrink_grid()), dim3(kShrinkThreads), (size_t)smem, st, 1u,
                    maps, a);
}

cudaError_t launch_sgmv_reduce(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *part,
                               float *buf, cudaStream_t st) {
  if (mv.num_tokens <= 0 || mv.num_slots <= 1) return cudaSuccess;
  SgReduceArgs a{};
  a.u.src = part;
  a.u.parts = 1;
  a.u.n_slices = d.n_slices;
  a.u.r_max = d.r_max;
  a.u.T = mv.num_tokens;
  a.buf = buf;
  a.work = mv.work;
  a.sorted_rows = mv.sorted_rows;
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
  a.err = const_cast<int32_t *>(mv.work) + WorkLists::kErrWord;
  a.L = list_of(mv, sel);
  a.shrink_grid = shrink_grid();
  a.nb = nb_of(d);
  a.maxp = maxp_of(mv.num_tokens, mv.num_slots, a.shrink_grid);
  return launch_pdl(sgmv_reduce_kernel, dim3((unsigned)(2 * sm_count())), dim3(kTileM), 0, st, 1u, a);
}

cudaError_t launch_sgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *u_src,
                               int u_parts, void *y, int64_t ldy, int y_dtype, cudaStream_t st, bool behind) {
  if (mv.num_tokens <= 0 || mv.num_slots <= 1) return cudaSuccess;
  const int kN = y_dtype == LORA_BF16 ? YCols<__nv_bfloat16>::kN : YCols<float>::kN;
  SgExpandMaps maps;
  memset(&maps, 0, sizeof(maps));
  int64_t width = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    cudaError_t e = make_map(&maps.b[s], d.B[s], (uint64_t)d.out_sizes[s], (uint64_t)d.r_max, (uint64_t)d.num_slots,
                             64u, (uint32_t)d.r_max, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    width += d.out_sizes[s];
  }
  cudaError_t em = make_rows_map(&maps.y, y, y_dtype == LORA_BF16, (uint64_t)width, (uint64_t)mv.num_tokens, ldy,
                                 y_dtype == LORA_BF16 ? 64u : 32u);
  if (em != cudaSuccess) return em;
  em = make_rows_map(&maps.ys, y, y_dtype == LORA_BF16, (uint64_t)width, (uint64_t)mv.num_tokens, ldy,
                     y_dtype == LORA_BF16 ? 64u : 32u, 32u);
  if (em != cudaSuccess) return em;
  SgExpandArgs a{};
  a.behind = behind ? 1 : 0;
  a.u.src = u_src;
  a.u.parts = u_parts;
  a.u.n_slices = d.n_slices;
  a.u.r_max = d.r_max;
  a.u.T = mv.num_tokens;
  a.y = y;
  a.ldy = ldy;
  a.work = mv.work;
  a.sorted_rows = mv.sorted_rows;
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
  a.err = const_cast<int32_t *>(mv.work) + WorkLists::kErrWord;
  a.L = list_of(mv, sel);
  a.shrink_grid = shrink_grid();
  a.nb = nb_of(d);
  a.maxp = maxp_of(mv.num_tokens, mv.num_slots, a.shrink_grid);
  int off = 0, nb = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    a.out_sizes[s] = d.out_sizes[s];
    a.out_off[s] = off;
    off += d.out_sizes[s];
    a.nb_start[s] = nb;
    nb += (d.out_sizes[s] + kN - 1) / kN;
  }
  a.nb_start[d.n_slices] = nb;
  a.nk = d.r_max > 64 ? 2 : 1;
  a.b_bytes = d.r_max * kN * 2;
  const int fixed = kAlignSlack + 512 + 2 * a.nk * kUKRegion;  // 512: barriers
  a.b_stages = 3;
  a.y_stages = 4;
  while (fixed + a.b_stages * a.b_bytes + a.y_stages * kYStage > kSmemMax && a.y_stages > 2) --a.y_stages;
  while (fixed + a.b_stages * a.b_bytes + a.y_stages * kYStage > kSmemMax && a.b_stages > 2) --a.b_stages;
  const int smem = fixed + a.b_stages * a.b_bytes + a.y_stages * kYStage;
  if (smem > kSmemMax) return cudaErrorInvalidValue;
  const void *k = y_dtype == LORA_BF16 ? (const void *)sgmv_expand_kernel<__nv_bfloat16>
                                       : (const void *)sgmv_expand_kernel<float>;
  cudaError_t e = set_max_dynamic_smem(k, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)sm_count());
  if (y_dtype == LORA_BF16)
    return launch_pdl(sgmv_expand_kernel<__nv_bfloat16>, grid, dim3(kExpandThreads), (size_t)smem, st, 1u, maps, a);
  return launch_pdl(sgmv_expand_kernel<float>, grid, dim3(kExpandThreads), (size_t)smem, st, 1u, maps, a);
}

}  // namespace ra
