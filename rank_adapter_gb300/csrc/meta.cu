// Token metadata (LoRAKernelMeta.prepare_tensors of the page "vLLM 源码完全拆解(十八):
// 多 LoRA 服务", section "LoRAKernelMeta:先按槽位排序"): a stable counting sort of
// token indices by slot, the segments present (ascending slot, with counts and
// start offsets that begin at 0), the no-LoRA flag, and the work lists the
// shrink / expand kernels read.
//
// One CTA (256 threads for small batches and tables, else 1024). Each warp
// owns a contiguous range of tokens and keeps a
// private histogram row in shared memory; a per-slot pass turns the histograms
// into exclusive per-(warp, slot) offsets; the scatter pass walks every warp's
// range in batch order and ranks equal slots inside each 32-token chunk with
// __match_any_sync. Warp ranges are in batch order, so the sort is stable and
// its result does not depend on scheduling.
#include "common.cuh"

namespace ra {
namespace {

constexpr int kSmallThreads = 256;  // batches of at most kSmallT tokens and tables of at most 256 slots
constexpr int kSmallT = 2048;
constexpr int kBigThreads = 1024;
constexpr int kCache = 8;            // 32-token chunks per warp whose slot ids stay in registers

struct MetaArgs {
  const int32_t *token_slot;
  int32_t T, S;
  int32_t *sorted_rows, *seg_slot, *seg_count, *seg_start, *num_segs, *no_lora, *status;
  int32_t *work;
  int early;  // the previous call's kernels do not read these outputs: write them without waiting
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix sums of N values per thread over the whole CTA, with one
// pair of barriers for all N. All threads call it.
template <int N, int kWarps>
__device__ void block_excl_scan_n(const int (&v)[N], int (&excl)[N], int (&total)[N], int *tmp /*[N][kWarps]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    incl[i] = warp_incl_scan(v[i]);
    if (lane == 31) tmp[i * kWarps + warp] = incl[i];
  }
  __syncthreads();
  if (warp == 0) {  // lanes past the warp count scan zeros and write nothing
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int w = warp_incl_scan(lane < kWarps ? tmp[i * kWarps + lane] : 0);
      if (lane < kWarps) tmp[i * kWarps + lane] = w;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    excl[i] = (warp > 0 ? tmp[i * kWarps + warp - 1] : 0) + incl[i] - v[i];
    total[i] = tmp[i * kWarps + kWarps - 1];
  }
  __syncthreads();
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads, 1) prepare_meta_kernel(MetaArgs a) {
  constexpr int kWarps = kThreads / 32;
  extern __shared__ int32_t sm[];
  const int S = a.S, T = a.T;
  const int hs = S + 1;             // odd row stride: a warp reading one slot's column hits 32 banks
  int32_t *hist = sm;                  // [kWarps][hs]: counts, then offsets inside each slot
  int32_t *tot_s = sm + kWarps * hs;   // [S] tokens per slot
  int32_t *base_s = tot_s + S;         // [S] first sorted row of each slot
  int32_t *rec_a = base_s + S;         // [S] int offset of the slot's record in the "all" list, or -1
  int32_t *rec_k = rec_a + S;          // [S] int offset of its record in the small or large list
  // (the slot-indexed copy of a slot's "all" record is at WorkLists::by_slot(S) + slot * kRec)
  __shared__ int tmp[7 * kWarps];
  __shared__ int s_bad;
  __shared__ int s_long;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Everything up to the merged scan reads only token_slot (complete when
  // this call was enqueued) and writes only shared memory, so it runs before
  // the wait, beside the tail of the previous kernel; the outputs, which
  // earlier kernels may still be reading, are written after it. The
  // successor is released at once: before its own wait it reads only the
  // slot table (a shrink starts streaming its A chunk).
  pdl_trigger();

  for (int i = tid; i < kWarps * hs; i += kThreads) hist[i] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // Pass 1: per-warp histograms over contiguous token ranges.
  const int per = (T + kWarps - 1) / kWarps;
  const int t0 = min(T, warp * per), t1 = min(T, t0 + per);
  int bad = 0;
  int cache[kCache];  // slot ids of this lane's first kCache chunks, for pass 2
#pragma unroll
  for (int c = 0; c < kCache; ++c) cache[c] = 0;
  for (int b = t0, c = 0; b < t1; b += 32, ++c) {
    const int t = b + lane;
    const bool valid = t < t1;
    int s = 0;
    if (valid) {
      s = a.token_slot[t];
      if (s < 0 || s >= S) { s = 0; ++bad; }
    }
#pragma unroll
    for (int cc = 0; cc < kCache; ++cc)
      if (cc == c) cache[cc] = s;
    const uint32_t act = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const uint32_t peers = __match_any_sync(act, s);
      if (lane == __ffs(peers) - 1) hist[warp * hs + s] += __popc(peers);
    }
    __syncwarp();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
  if (lane == 0 && bad) atomicAdd(&s_bad, bad);
  __syncthreads();

  // Per slot, across the kWarps warp rows: exclusive offsets (one warp scan per slot).
  if (tid == 0) s_long = 0;
  __syncthreads();
  for (int s = warp; s < S; s += kWarps) {
    const int c = lane < kWarps ? hist[lane * hs + s] : 0;
    const int incl = warp_incl_scan(c);
    if (lane < kWarps) hist[lane * hs + s] = incl - c;
    if (lane == 31) {
      tot_s[s] = incl;
      if (s != 0 && incl >= LORA_AUTO_LONG_ROWS) s_long = 1;  // a long LoRA segment exists
    }
  }
  __syncthreads();

  // One merged scan: slot bases, segment / list indices and tile offsets.
  const int tot = tid < S ? tot_s[tid] : 0;
  const bool present = tid < S && tot > 0;
  const bool lora = present && tid != 0;
  // AUTO's split: segments of LORA_SGMV_MIN_ROWS or more go to the large
  // list only when the batch holds a segment of LORA_AUTO_LONG_ROWS or more
  // (a prefill chunk); otherwise every segment is small (all on BGMV).
  const bool large = lora && tot >= LORA_SGMV_MIN_ROWS && s_long != 0;
  const bool small = lora && !large;
  const int tiles = lora ? (tot + LORA_SGMV_TILE_M - 1) / LORA_SGMV_TILE_M : 0;
  const int vals[7] = {tot, present, lora, small, large, tiles, large ? tiles : 0};
  int ex[7], tl[7];
  block_excl_scan_n<7, kWarps>(vals, ex, tl, tmp);
  const int base = ex[0], seg_idx = ex[1];
  const int nsegs = tl[1], n_all = tl[2], n_small = tl[3], n_large = tl[4];
  const int tiles_all = tl[5], tiles_large = tl[6];
  constexpr int R = WorkLists::kRec;

  int32_t *W = a.work;
  if (tid < S) {
    base_s[tid] = base;
    rec_a[tid] = lora ? WorkLists::list(S, kListAll) + ex[2] * R : -1;
    rec_k[tid] = small ? WorkLists::list(S, kListSmall) + ex[3] * R
               : large ? WorkLists::list(S, kListLarge) + ex[4] * R : -1;
  }
  // The outputs may still be read by the kernels of the previous call; with
  // `early` the caller has promised they are not (another metadata buffer),
  // and the wait moves to the kernel's exit.
  if (!a.early) pdl_wait();
  if (tid < S) {
    W[WorkLists::slot_rec(S, kListAll) + tid] = lora ? ex[2] : -1;
    W[WorkLists::slot_rec(S, kListSmall) + tid] = small ? ex[3] : -1;
    W[WorkLists::slot_rec(S, kListLarge) + tid] = large ? ex[4] : -1;
  }
  if (present) {
    a.seg_slot[seg_idx] = tid;
    a.seg_count[seg_idx] = tot;
    a.seg_start[seg_idx] = base;
  }
  if (lora) {
    const int4 head = make_int4(seg_idx, tid, tot, base);
    const int4 none = make_int4(-1, -1, -1, -1);
    int32_t *ra_ = W + WorkLists::list(S, kListAll) + ex[2] * R;
    int32_t *rk_ = W + (small ? WorkLists::list(S, kListSmall) + ex[3] * R : WorkLists::list(S, kListLarge) + ex[4] * R);
    reinterpret_cast<int4 *>(ra_)[0] = head;
    reinterpret_cast<int4 *>(ra_)[1] = none;
    reinterpret_cast<int4 *>(rk_)[0] = head;
    reinterpret_cast<int4 *>(rk_)[1] = none;
    int32_t *rs_ = W + WorkLists::by_slot(S) + tid * R;
    reinterpret_cast<int4 *>(rs_)[0] = head;
    reinterpret_cast<int4 *>(rs_)[1] = none;
    W[WorkLists::all_tile_start(S) + ex[2]] = ex[5];
    if (large) W[WorkLists::large_tile_start(S) + ex[4]] = ex[6];
  }
  // Unused records, tails, scalars.
  const int4 none = make_int4(-1, -1, -1, -1);
  if (tid < S && !lora) {
    reinterpret_cast<int4 *>(W + WorkLists::by_slot(S) + tid * R)[0] = none;
    reinterpret_cast<int4 *>(W + WorkLists::by_slot(S) + tid * R)[1] = none;
  }
  for (int i = tid; i < S; i += kThreads) {
    if (i >= n_all) {
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListAll) + i * R)[0] = none;
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListAll) + i * R)[1] = none;
    }
    if (i >= n_small) {
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListSmall) + i * R)[0] = none;
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListSmall) + i * R)[1] = none;
    }
    if (i >= n_large) {
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListLarge) + i * R)[0] = none;
      reinterpret_cast<int4 *>(W + WorkLists::list(S, kListLarge) + i * R)[1] = none;
    }
  }
  for (int i = tid; i <= S; i += kThreads) {
    if (i < S && i >= nsegs) { a.seg_slot[i] = -1; a.seg_count[i] = 0; }
    if (i >= nsegs) a.seg_start[i] = T;
    if (i >= n_all) W[WorkLists::all_tile_start(S) + i] = tiles_all;
    if (i >= n_large) W[WorkLists::large_tile_start(S) + i] = tiles_large;
  }
  if (tid == 0) {
    W[0] = n_all; W[1] = n_small; W[2] = n_large; W[3] = tiles_all; W[4] = tiles_large;
    W[5] = 0; W[6] = 0; W[7] = 0;
    *a.num_segs = nsegs;
    *a.status = s_bad;
    *a.no_lora = (T - tot == 0) ? 1 : 0;   // thread 0 holds the slot-0 count
  }
  __syncthreads();

  // Pass 2: stable scatter of token indices; the first 4 rows of each LoRA
  // segment also go into its unit records.
  for (int b = t0, c = 0; b < t1; b += 32, ++c) {
    const int t = b + lane;
    const bool valid = t < t1;
    int s = 0;
    if (valid) {
      if (c < kCache) {
#pragma unroll
        for (int cc = 0; cc < kCache; ++cc)
          if (cc == c) s = cache[cc];
      } else {
        s = a.token_slot[t];
        if (s < 0 || s >= S) s = 0;
      }
    }
    const uint32_t act = __ballot_sync(0xffffffffu, valid);
    uint32_t peers = 0;
    if (valid) {
      peers = __match_any_sync(act, s);
      const int rel = hist[warp * hs + s] + __popc(peers & lanemask_lt());
      a.sorted_rows[base_s[s] + rel] = t;
      if (rel < 4 && rec_a[s] >= 0) {
        W[rec_a[s] + 4 + rel] = t;
        W[rec_k[s] + 4 + rel] = t;
        W[WorkLists::by_slot(S) + s * WorkLists::kRec + 4 + rel] = t;
      }
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) hist[warp * hs + s] += __popc(peers);
    __syncwarp();
  }
  if (a.early) pdl_wait();  // this kernel's completion still implies its predecessors'
}

}  // namespace

cudaError_t launch_prepare_meta(const lora_meta &m, cudaStream_t st, bool early) {
  MetaArgs a;
  a.early = early ? 1 : 0;
  a.token_slot = m.token_slot;
  a.T = m.num_tokens;
  a.S = m.num_slots;
  a.sorted_rows = m.sorted_rows;
  a.seg_slot = m.seg_slot;
  a.seg_count = m.seg_count;
  a.seg_start = m.seg_start;
  a.num_segs = m.num_segs;
  a.no_lora = m.no_lora;
  a.status = m.status;
  a.work = static_cast<int32_t *>(m.tiles);
  const bool small = m.num_tokens <= kSmallT && m.num_slots <= kSmallThreads;
  const int nt = small ? kSmallThreads : kBigThreads;
  void (*k)(MetaArgs) = small ? prepare_meta_kernel<kSmallThreads> : prepare_meta_kernel<kBigThreads>;
  const size_t smem = ((size_t)(nt / 32) * (m.num_slots + 1) + 4 * (size_t)m.num_slots) * sizeof(int32_t);
  cudaError_t e = set_max_dynamic_smem((const void *)k, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(1), dim3(nt), smem, st, 1u, a);
}

}  // namespace ra
