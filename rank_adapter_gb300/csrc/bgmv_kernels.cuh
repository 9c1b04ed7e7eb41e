// Device side of the BGMV family (kernel templates and their helpers),
// shared by the translation units that instantiate them (bgmv_shrink_k.cu
// and bgmv_expand_k.cu compile in parallel); bgmv.cu holds the host side
// (geometry, dispatch).
//
// BGMV shrink / expand on CUDA cores: the decode form of the multi-LoRA delta
// (handbook page "多 LoRA 服务：分段矩阵乘与适配器调度", section "不合并权重，批量计算":
// each token gathers its own adapter and does a small matrix-vector product).
//
// Decode is bound by reading each active adapter's A and B once from HBM
// (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section "成本与边界": about
// 2 r (d_in + d_out) extra elements per layer), so the kernels are organised
// around the weights, in small uniform CTAs that keep every SM streaming:
//
// * shrink: one CTA per (segment, slice, chunk of d_in rows of 32 KB of A).
//   All of its A rows and the matching x columns of the tile's 4 tokens are
//   requested at once with 16-byte cp.async copies; a thread feeds a
//   16-byte weight vector to the tile's tokens with mixed-precision FMAs
//   (bf16 products, fp32 sums; packed fp32x2 FMAs for fp32 tables); row
//   groups combine by a recursive-halving shuffle reduce-scatter
//   and a fixed-order sum over warps. It writes unscaled partial rows to a
//   caller-provided workspace (or, for lora_shrink with a single chunk, the
//   scaled rank-r rows u = s * x A directly).
// * expand: one CTA per (segment, slice, column chunk of 32 KB of B). It
//   forms u by summing the chunk partials in chunk order (or reads u), then
//   adds u B into y with packed FMAs over pairs of rank indices. Where the
//   chunk is narrower than the block (high ranks), thread groups take
//   several token tiles of a unit at once.
// * reduce: for the split path, turns the partials into the u buffer with
//   the same arithmetic, so shrink + expand and the fused apply (shrink +
//   expand-from-partials, two launches) give bitwise identical results.
#pragma once

#include <utility>

#include "common.cuh"

namespace ra {
namespace bgmvk {


constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Shrink CTAs are smaller (128 threads, ~43 KB) so that five fit on an SM and a
// decode batch's whole shrink grid is resident at once: every A chunk is then
// requested at kernel start, before the metadata wait.
constexpr int kSThreads = 128;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSMinBlocks = 5;
constexpr int kTT = 4;               // tokens per tile
constexpr int kAStageBytes = 16384;  // A bytes per stretch
constexpr int kStretches = 2;        // stretches per shrink CTA (all in flight at once)
constexpr int kBPassBytes = 32768;   // B bytes per expand CTA (twice that for deep grids, see kWideGrid)
// An expand grid of more CTAs than this at kBPassBytes (about 2.2 waves of
// three CTAs per SM on 152 SMs) takes CTAs of twice the columns: for a
// vocabulary-wide output that measured 110 -> 92 us, for the MoE step's
// 2048-CTA grids 125 -> 120 us and for the mixed batch's 83 -> 80 us, while
// shallow decode grids are faster with the narrower CTAs (fewer CTAs would
// leave SMs idle; 512 here made the 32-layer step 1% slower).
constexpr int kWideGrid = 1024;
constexpr int kSmallTable = 256;     // slot tables up to this size: rank / scale copied whole
constexpr int kRowsWin = 32;         // token rows of a unit kept in shared memory (a sliding window)
constexpr int kKCReg = 4;            // expand: chunk partials of the next tile held in registers (d_in up to 4 chunks)
constexpr int kExpandNG = 4;         // expand: most token tiles of a unit run side by side
constexpr int kReach = kThreads * 4; // expand: columns one tile pass of the whole block covers

struct Geo {
  int d_in, r_max;
  int sc;                 // A rows per stretch (multiple of 8)
  int kchunk, kc_count;   // d_in rows per shrink CTA, and chunks per unit
  int pw;                 // B columns per expand CTA (multiple of 8)
  int a_stage, x_stage;   // bytes of the A and x parts of one stretch buffer
  int off_rs, off_rows, off_u, off_ring, off_red, off_b;
  int smem_shrink, smem_expand, smem_reduce;
};

struct BgmvArgs {
  const void *x;
  int64_t ldx;
  int x_div;            // LoRA row i reads x row i / x_div
  const void *A[LORA_MAX_SLICES];
  const void *B[LORA_MAX_SLICES];
  float *buf;           // shrink (to_parts == 0) and reduce: receives u rows
  float *part;          // shrink (to_parts == 1): receives chunk partials
  int to_parts;
  const float *u_in;    // expand / reduce: chunk partials or u rows
  int u_parts;          // expand: u_in holds chunk partials
  void *y;
  int64_t ldy;
  int out_sizes[LORA_MAX_SLICES];
  int out_off[LORA_MAX_SLICES];
  int slice_order[LORA_MAX_SLICES];      // slices by decreasing width: heavy units launch first
  int chunk_start[LORA_MAX_SLICES + 1];  // expand: column chunks per slice
  int n_slices, max_items;
  MetaView mv;
  int list;      // int offset of the unit-record list inside the work lists
  int by_slot;   // shrink: grid rows are slots 1..S-1 (A prefetched before the wait)
  int small_only;  // by_slot on the short-segment list: skip slots whose segment is long
  int wave;      // by_slot shrink grids deeper than one wave: CTAs resident at once (else 0)
  int pre;       // expand: runs right behind this library's shrink / reduce
  const int32_t *slot_rank;
  const float *slot_scale;
  Geo g;
};

struct Unit {
  int slot, cnt, start, r_a;
  float scale;
};

// One unit record (segment, slot, count, start, first rows) plus the slot's
// rank and scale, in one round trip: small slot tables are copied whole into
// shared memory in parallel with the record. The first rows go to rows[].
// Returns false (uniformly over the CTA) for an unused record.
__device__ __forceinline__ bool load_unit(const BgmvArgs &a, int item, Unit &u, unsigned char *smem, int *rows) {
  const int S = a.mv.num_slots;
  const bool small_table = S <= kSmallTable;
  int32_t *rank_s = reinterpret_cast<int32_t *>(smem + a.g.off_rs);
  float *scale_s = reinterpret_cast<float *>(rank_s + kSmallTable);
  if (small_table) {
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
      rank_s[i] = a.slot_rank[i];
      scale_s[i] = a.slot_scale[i];
    }
  }
  const int4 *rec = reinterpret_cast<const int4 *>(a.mv.work + a.list + item * WorkLists::kRec);
  const int4 h = rec[0], r = rec[1];
  if (h.y < 0) return false;
  u.slot = h.y;
  u.cnt = h.z;
  u.start = h.w;
  if (threadIdx.x < kTT)
    rows[threadIdx.x] = threadIdx.x == 0 ? r.x : threadIdx.x == 1 ? r.y : threadIdx.x == 2 ? r.z : r.w;
  __syncthreads();
  const int rk = small_table ? rank_s[u.slot] : a.slot_rank[u.slot];
  u.r_a = min(max(rk, 0), a.g.r_max);
  u.scale = small_table ? scale_s[u.slot] : a.slot_scale[u.slot];
  return true;
}

// Widen bf16 / fp32 weights to fp32.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename TW>
__device__ __forceinline__ void widen16(const uint4 &q, float *f) {
  if constexpr (sizeof(TW) == 2) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf_lo(w[i]);
      f[2 * i + 1] = bf_hi(w[i]);
    }
  } else {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
  }
}
// Two consecutive elements of a row as fp32.
template <typename T>
__device__ __forceinline__ float2 load2(const T *p) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
    return make_float2(bf_lo(w), bf_hi(w));
  } else {
    return *reinterpret_cast<const float2 *>(p);
  }
}
// Four consecutive elements of a row as fp32, and back.
template <typename T>
__device__ __forceinline__ void load4(const T *p, float *f) {
  if constexpr (sizeof(T) == 2) {
    const uint2 q = *reinterpret_cast<const uint2 *>(p);
    f[0] = bf_lo(q.x); f[1] = bf_hi(q.x); f[2] = bf_lo(q.y); f[3] = bf_hi(q.y);
  } else {
    const float4 q = *reinterpret_cast<const float4 *>(p);
    f[0] = q.x; f[1] = q.y; f[2] = q.z; f[3] = q.w;
  }
}
template <typename T>
__device__ __forceinline__ void store4(T *p, const float *f) {
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(f[0], f[1]), hi = __floats2bfloat162_rn(f[2], f[3]);
    uint2 q;
    q.x = *reinterpret_cast<uint32_t *>(&lo);
    q.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = q;
  } else {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
}

// acc += (lo(w), hi(w)) * x for a word w holding two bf16 values and a bf16
// x: two mixed-precision FMAs (bf16 products, fp32 accumulation, one rounding
// each: the same result as an fp32 FMA of the widened operands).
__device__ __forceinline__ void fma2_bf16(uint32_t w, uint16_t x, float2 &acc) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.bf16 %0, lo, %3, %0;\n\t"
      "fma.rn.f32.bf16 %1, hi, %3, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w), "h"(x));
}

// Four consecutive y values as loaded (bf16 bits or fp32), widened later.
template <typename T> struct YRaw;
template <> struct YRaw<__nv_bfloat16> {
  uint2 q;
  __device__ static __forceinline__ YRaw load(const __nv_bfloat16 *p) { return {*reinterpret_cast<const uint2 *>(p)}; }
  __device__ __forceinline__ void to_f(float *f) const {
    f[0] = bf_lo(q.x); f[1] = bf_hi(q.x); f[2] = bf_lo(q.y); f[3] = bf_hi(q.y);
  }
};
template <> struct YRaw<float> {
  float4 q;
  __device__ static __forceinline__ YRaw load(const float *p) { return {*reinterpret_cast<const float4 *>(p)}; }
  __device__ __forceinline__ void to_f(float *f) const { f[0] = q.x; f[1] = q.y; f[2] = q.z; f[3] = q.w; }
};

// Sum N values per lane over the lanes that share bits [0, log2(NV)) of the
// lane id (recursive halving). Afterwards the lane keeps max(1, N / (32 / NV))
// sums in vals[0..), whose positions in the original array start at the
// returned offset. When the lanes outnumber the values (N < 32 / NV), the
// levels left after the last halving add the single remaining value across
// lanes (butterfly), so the lanes that end up with the same position hold
// the same complete sum.
template <int N, int NV>
__device__ __forceinline__ int reduce_scatter(float (&vals)[N]) {
  const int lane = threadIdx.x & 31;
  int off = 0;
#pragma unroll
  for (int lvl = 0, o = NV; o < 32; ++lvl, o <<= 1) {
    const int half = (N >> lvl) >> 1;
    if (half == 0) {
      vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], o);
      continue;
    }
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      if (i < half) {
        const float send = up ? vals[i] : vals[i + half];
        const float keep = up ? vals[i + half] : vals[i];
        vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    if (up) off += half;
  }
  return off;
}

// B rows 0..nrows-1, columns [pc0, pc0 + pcn) of one slot -> Bs (row stride pw). A warp per row.
template <typename TW>
__device__ __forceinline__ void issue_b(TW *Bs, int pw, const TW *Bslot, int out_s, int nrows, int pc0, int pcn) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int upr = pcn * (int)sizeof(TW) / 16;
  for (int k = warp; k < nrows; k += kWarps) {
    const char *src = reinterpret_cast<const char *>(Bslot + (int64_t)k * out_s + pc0);
    char *dst = reinterpret_cast<char *>(Bs + k * pw);
    for (int c = lane; c < upr; c += 32) cp_async16(dst + c * 16, src + c * 16);
  }
}

// y[rows[t], col_base + c] += sum_k u[t][k] B[k][c] for tokens t < nt and
// columns [0, pcn) of a staged pass. Bs holds B rows 0..r_pad-1 (r_pad = r_a
// rounded up to even; an extra row is zero); us is u as [kTT][r_max] with the
// rank tail and absent tokens zero. Thread lt of a group of GS threads takes
// columns 4 lt, 4 (lt + GS), ...; pairs of k in the two lanes of packed FMAs.
template <typename TW, typename TY, int GS, int NT>
__device__ __forceinline__ void expand_pass_nt(const TW *Bs, int pw, const float *us, int r_max, int r_pad,
                                               const int *rows, int rbase, TY *y, int64_t ldy, int col_base,
                                               int pcn, int lt) {
  for (int cq = lt * 4; cq < pcn; cq += GS * 4) {
    // The y values are requested before the products so that their latency
    // overlaps the FMAs (kept as loaded: 8 or 16 bytes per token).
    YRaw<TY> yr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) yr[t] = YRaw<TY>::load(y + (int64_t)rows[(rbase + t) % kRowsWin] * ldy + col_base + cq);
    float2 acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[t][c] = make_float2(0.f, 0.f);
    const TW *bp = Bs + cq;
#pragma unroll 2
    for (int k = 0; k < r_pad; k += 2) {
      float b0[4], b1[4];
      load4(bp + k * pw, b0);
      load4(bp + (k + 1) * pw, b1);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float2 u2 = *reinterpret_cast<const float2 *>(us + t * r_max + k);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[t][c] = __ffma2_rn(u2, make_float2(b0[c], b1[c]), acc[t][c]);
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float yv[4];
      yr[t].to_f(yv);
#pragma unroll
      for (int c = 0; c < 4; ++c) yv[c] += acc[t][c].x + acc[t][c].y;
      store4(y + (int64_t)rows[(rbase + t) % kRowsWin] * ldy + col_base + cq, yv);
    }
  }
}
// The tile's nt (1..kTT) tokens; every output takes the same arithmetic whatever nt is.
template <typename TW, typename TY, int GS>
__device__ __forceinline__ void expand_pass(const TW *Bs, int pw, const float *us, int r_max, int r_pad,
                                            const int *rows, int rbase, int nt, TY *y, int64_t ldy, int col_base,
                                            int pcn, int lt) {
  if (nt >= 4) expand_pass_nt<TW, TY, GS, 4>(Bs, pw, us, r_max, r_pad, rows, rbase, y, ldy, col_base, pcn, lt);
  else if (nt == 3) expand_pass_nt<TW, TY, GS, 3>(Bs, pw, us, r_max, r_pad, rows, rbase, y, ldy, col_base, pcn, lt);
  else if (nt == 2) expand_pass_nt<TW, TY, GS, 2>(Bs, pw, us, r_max, r_pad, rows, rbase, y, ldy, col_base, pcn, lt);
  else expand_pass_nt<TW, TY, GS, 1>(Bs, pw, us, r_max, r_pad, rows, rbase, y, ldy, col_base, pcn, lt);
}

// The arithmetic of one shrink tile of up to 4 tokens. With NVE lanes per A
// row (the slot's rank rounded up to whole 16-byte vectors, then to a power
// of two: a low-rank slot puts its threads on more row groups instead of
// idle lanes), thread (row group rq, vector v) accumulates, for every token t
// of the tile, the products of its A rows with the token's x columns, rows in
// increasing order within each stretch, packed fp32x2 FMAs.
template <typename TW, int NVE>
struct TileMath {
  static constexpr int VEC = Elem<TW>::kVec;
  static constexpr int NRG = kSThreads / NVE;  // row groups
  static constexpr int NVAL = kTT * VEC;       // accumulators per thread
  static constexpr int LPV = 32 / NVE;         // lanes sharing one vector column
  static constexpr int NKEEP = NVAL / (LPV > NVAL ? NVAL : LPV);

  // acc2[t * VEC / 2 + p] = (acc[t][2p], acc[t][2p + 1]) over the chunk's nst stretches,
  // for the NT tokens the tile holds (the other entries stay zero).
  template <int NT>
  __device__ static __forceinline__ void products_nt(const Geo &g, unsigned char *smem, int nva, int klen, int nst,
                                                     float2 (&acc2)[NVAL / 2]) {
    const int tid = threadIdx.x;
    const int v = tid % NVE, rq = tid / NVE;
#pragma unroll
    for (int i = 0; i < NVAL / 2; ++i) acc2[i] = make_float2(0.f, 0.f);
    for (int s = 0; s < nst; ++s) {
      if (v < nva) {
        const int nr = min(g.sc, klen - s * g.sc);
        const TW *As = reinterpret_cast<const TW *>(smem + g.off_ring + s * (g.a_stage + g.x_stage)) + v * VEC;
        const TW *xs = reinterpret_cast<const TW *>(smem + g.off_ring + s * (g.a_stage + g.x_stage) + g.a_stage);
        if constexpr (sizeof(TW) == 2) {
          // bf16 operands straight into mixed-precision FMAs (one rounding, as
          // an fp32 FMA of the widened values): no widening instructions.
          const uint16_t *xr = reinterpret_cast<const uint16_t *>(xs);
#pragma unroll 4
          for (int j = rq; j < nr; j += NRG) {
            const uint4 q = *reinterpret_cast<const uint4 *>(As + j * g.r_max);
            const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint16_t xt = xr[t * g.sc + j];
#pragma unroll
              for (int p = 0; p < VEC / 2; ++p) fma2_bf16(wq[p], xt, acc2[t * (VEC / 2) + p]);
            }
          }
        } else {
#pragma unroll 4
          for (int j = rq; j < nr; j += NRG) {
            float w[VEC];
            widen16<TW>(*reinterpret_cast<const uint4 *>(As + j * g.r_max), w);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const float xt = Elem<TW>::to_f(xs[t * g.sc + j]);
              const float2 xx = make_float2(xt, xt);
#pragma unroll
              for (int p = 0; p < VEC / 2; ++p)
                acc2[t * (VEC / 2) + p] = __ffma2_rn(xx, make_float2(w[2 * p], w[2 * p + 1]), acc2[t * (VEC / 2) + p]);
            }
          }
        }
      }
    }
  }
  // The tile's nt (1..kTT) tokens: each token's products are the same whatever nt is.
  __device__ static __forceinline__ void products(const Geo &g, unsigned char *smem, int nva, int klen, int nst,
                                                  int nt, float2 (&acc2)[NVAL / 2]) {
    static_assert(kTT == 4, "products dispatches tiles of up to 4 tokens");
    if (nt >= 4) products_nt<4>(g, smem, nva, klen, nst, acc2);
    else if (nt == 3) products_nt<3>(g, smem, nva, klen, nst, acc2);
    else if (nt == 2) products_nt<2>(g, smem, nva, klen, nst, acc2);
    else products_nt<1>(g, smem, nva, klen, nst, acc2);
  }

  // Row groups (in-warp recursive halving) into the per-warp rows wred
  // [kSWarps][kTT][r_max]. Entries of absent tokens carry garbage and are
  // never read back.
  __device__ static __forceinline__ void to_warp_rows(const Geo &g, float *wred, float2 (&acc2)[NVAL / 2]) {
    const int tid = threadIdx.x, warp = tid >> 5, v = tid % NVE;
    float acc[NVAL];
#pragma unroll
    for (int i = 0; i < NVAL / 2; ++i) {
      acc[2 * i] = acc2[i].x;
      acc[2 * i + 1] = acc2[i].y;
    }
    const int off = reduce_scatter<NVAL, NVE>(acc);
#pragma unroll
    for (int i = 0; i < NKEEP; ++i) {
      const int idx = off + i, t = idx / VEC, e = idx % VEC;
      wred[(warp * kTT + t) * g.r_max + v * VEC + e] = acc[i];
    }
  }
};

// The CTA's chunk sum for entry i = t * r_max + k of a tile: the warps' rows in warp order.
__device__ __forceinline__ float warp_rows_sum(const float *wred, int r_max, int i) {
  float sum = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kSWarps; ++w2) sum += wred[w2 * kTT * r_max + i];
  return sum;
}

// Shrink. Grid: (max_items * n_slices, kc_count); block (b, c) -> unit
// (slice_order[b / max_items], item b % max_items), rows [c * kchunk, +kchunk).
// The token tiles of one shrink unit, with NVE lanes per A row (TileMath).
template <typename TW, int NVE>
__device__ __forceinline__ void shrink_tiles(const BgmvArgs &a, unsigned char *smem, int *rows, const Unit &u,
                                             int slice, int kc, int k0, int klen, int nst) {
  using M = TileMath<TW, NVE>;
  constexpr int VEC = Elem<TW>::kVec;
  const Geo &g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r_max = g.r_max;
  const TW *x = static_cast<const TW *>(a.x);
  float *wred = reinterpret_cast<float *>(smem + g.off_red);  // [kSWarps][kTT][r_max]
  auto stX = [&](int b) {
    return reinterpret_cast<TW *>(smem + g.off_ring + b * (g.a_stage + g.x_stage) + g.a_stage);
  };
  const int nva = (u.r_a + VEC - 1) / VEC;
  const int ntiles = (u.cnt + kTT - 1) / kTT;
  // Token i of the unit is row rows[i % kRowsWin]. The x columns of a tile
  // are requested as soon as the previous tile's products are done, so their
  // latency overlaps that tile's reduction and stores.
  auto issue_x = [&](int tile) {
    const int nt = min(kTT, u.cnt - tile * kTT);
    for (int s = 0; s < nst; ++s) {
      const int r0 = s * g.sc, nr = min(g.sc, klen - r0);
      const int upr = nr / VEC;
      TW *xs = stX(s);
      for (int t = warp; t < nt; t += kSWarps) {
        const int row = rows[(tile * kTT + t) % kRowsWin];
        const TW *xsrc = x + (int64_t)(a.x_div == 1 ? row : row / a.x_div) * a.ldx + k0 + r0;
        for (int c = tid & 31; c < upr; c += 32) cp_async16(xs + t * g.sc + c * VEC, xsrc + c * VEC);
      }
    }
    cp_async_commit();
  };
  issue_x(0);  // rows 0..kTT-1 came with the unit record
  for (int i = kTT + tid; i < min(u.cnt, kRowsWin); i += kSThreads) rows[i] = a.mv.sorted_rows[u.start + i];
  for (int tile = 0; tile < ntiles; ++tile) {
    const int nt = min(kTT, u.cnt - tile * kTT);
    cp_async_wait_upto(0);
    __syncthreads();  // this tile's x, the A chunk and the token rows are in shared memory
    float2 acc2[M::NVAL / 2];
    M::products(g, smem, nva, klen, nst, nt, acc2);
    __syncthreads();  // every thread is done with the x stage
    const int nxt = tile + 1;
    const bool next_in_window = nxt < ntiles && (nxt * kTT) % kRowsWin != 0;
    if (next_in_window) issue_x(nxt);
    M::to_warp_rows(g, wred, acc2);
    __syncthreads();
    for (int i = tid; i < nt * r_max; i += kSThreads) {
      const int t = i / r_max, k = i - t * r_max;
      const float sum = warp_rows_sum(wred, r_max, i);
      if (!a.to_parts) {
        a.buf[((int64_t)slice * a.mv.num_tokens + rows[(tile * kTT + t) % kRowsWin]) * r_max + k] =
            k < u.r_a ? u.scale * sum : 0.f;
      } else {
        const int64_t pos = (int64_t)slice * a.mv.num_tokens + u.start + tile * kTT + t;
        a.part[(pos * g.kc_count + kc) * r_max + k] = sum;
      }
    }
    if (nxt < ntiles && !next_in_window) {  // the next tile starts a new window of token rows
      __syncthreads();
      for (int i = tid; i < kRowsWin && nxt * kTT + i < u.cnt; i += kSThreads)
        rows[i] = a.mv.sorted_rows[u.start + nxt * kTT + i];
      __syncthreads();
      issue_x(nxt);
    }
  }
}

template <typename TW, int NV>
__global__ void __launch_bounds__(kSThreads, kSMinBlocks) bgmv_shrink_kernel(BgmvArgs a) {
  constexpr int VEC = Elem<TW>::kVec;
  extern __shared__ __align__(16) unsigned char smem[];
  const Geo &g = a.g;
  const int kc = blockIdx.y;
  const int rows_per = a.by_slot ? a.mv.num_slots - 1 : a.max_items;
  const int slice = a.slice_order[blockIdx.x / rows_per];
  int *rows = reinterpret_cast<int *>(smem + g.off_rows);
  const int tid = threadIdx.x;
  const int r_max = g.r_max;
  const int k0 = kc * g.kchunk;
  const int klen = min(g.kchunk, g.d_in - k0);
  const int nst = (klen + g.sc - 1) / g.sc;  // stretches of this chunk (<= kStretches)
  auto stA = [&](int b) { return reinterpret_cast<TW *>(smem + g.off_ring + b * (g.a_stage + g.x_stage)); };
  // All A stretches of this chunk in flight at once, rank tail skipped.
  auto issue_a = [&](int slot, int nva) {
    const TW *Aslot = static_cast<const TW *>(a.A[slice]) + ((int64_t)slot * g.d_in + k0) * r_max;
    for (int s = 0; s < nst; ++s) {
      const int r0 = s * g.sc, nr = min(g.sc, klen - r0);
      const uint4 *src = reinterpret_cast<const uint4 *>(Aslot + (int64_t)r0 * r_max);
      uint4 *dst = reinterpret_cast<uint4 *>(stA(s));
      for (int i = tid; i < nr * NV; i += kSThreads)
        if ((i & (NV - 1)) < nva) cp_async16(dst + i, src + i);
    }
    cp_async_commit();
  };
  Unit u;
  if (a.by_slot) {
    // The slot table is complete before any kernel of this library starts
    // (see pdl_wait), so this slot's A chunk streams in while the metadata
    // kernel may still be running.
    u.slot = 1 + (int)blockIdx.x % rows_per;
    u.r_a = min(max(a.slot_rank[u.slot], 0), r_max);
    u.scale = a.slot_scale[u.slot];
    issue_a(u.slot, (u.r_a + VEC - 1) / VEC);
    if (a.wave > 0 && tid == 0) {
      // A grid deeper than one wave: the CTA one wave later in launch order
      // starts only as a CTA of this wave leaves, so this one brings that
      // CTA's A chunk (a full-rank slot's, one contiguous block) into L2 now.
      const int b2 = (int)(blockIdx.y * gridDim.x + blockIdx.x) + a.wave;
      if (b2 < (int)(gridDim.x * gridDim.y)) {
        const int x2 = b2 % (int)gridDim.x, kc2 = b2 / (int)gridDim.x;
        const int slot2 = 1 + x2 % rows_per;
        if (a.slot_rank[slot2] >= r_max) {
          const int k02 = kc2 * g.kchunk, klen2 = min(g.kchunk, g.d_in - k02);
          const TW *src = static_cast<const TW *>(a.A[a.slice_order[x2 / rows_per]]) + ((int64_t)slot2 * g.d_in + k02) * r_max;
          prefetch_l2(src, (uint32_t)(klen2 * r_max * (int)sizeof(TW)));
        }
      }
    }
    pdl_wait();
    pdl_trigger();
    // The slot-indexed copy of the slot's record: one load, no index lookup.
    const int4 *rec = reinterpret_cast<const int4 *>(a.mv.work + WorkLists::by_slot(a.mv.num_slots) +
                                                     u.slot * WorkLists::kRec);
    const int in_small = a.small_only ? a.mv.work[WorkLists::slot_rec(a.mv.num_slots, kListSmall) + u.slot] : 0;
    const int4 h = rec[0], r = rec[1];
    if (h.y < 0 || in_small < 0) {  // no tokens here (or the segment is on the other family's list)
      cp_async_wait_upto(0);
      return;
    }
    u.cnt = h.z;
    u.start = h.w;
    if (threadIdx.x < kTT)
      rows[threadIdx.x] = threadIdx.x == 0 ? r.x : threadIdx.x == 1 ? r.y : threadIdx.x == 2 ? r.z : r.w;
    __syncthreads();
  } else {
    pdl_wait();
    pdl_trigger();
    if (!load_unit(a, (int)blockIdx.x % rows_per, u, smem, rows)) return;
    issue_a(u.slot, (u.r_a + VEC - 1) / VEC);
  }
  int nve = 1;  // lanes per A row this unit needs (a power of two <= NV)
  while (nve < NV && nve * VEC < u.r_a) nve <<= 1;
  if (nve >= NV) shrink_tiles<TW, NV>(a, smem, rows, u, slice, kc, k0, klen, nst);
  else if constexpr (NV >= 2) {
    if (nve * 2 >= NV) shrink_tiles<TW, (NV >= 2 ? NV / 2 : 1)>(a, smem, rows, u, slice, kc, k0, klen, nst);
    else if constexpr (NV >= 4) {
      if (nve * 4 >= NV) shrink_tiles<TW, (NV >= 4 ? NV / 4 : 1)>(a, smem, rows, u, slice, kc, k0, klen, nst);
      else if constexpr (NV >= 8) {
        if (nve * 8 >= NV) shrink_tiles<TW, (NV >= 8 ? NV / 8 : 1)>(a, smem, rows, u, slice, kc, k0, klen, nst);
        else shrink_tiles<TW, (NV >= 16 ? NV / 16 : 1)>(a, smem, rows, u, slice, kc, k0, klen, nst);
      }
    }
  }
}

// u[t][k] of token `pos` (sorted position) from the chunk partials, summed in chunk order.
__device__ __forceinline__ float u_from_partials(const BgmvArgs &a, int slice, int pos, int k, const Unit &u) {
  if (k >= u.r_a) return 0.f;
  const float *p = a.u_in + (((int64_t)slice * a.mv.num_tokens + pos) * a.g.kc_count) * a.g.r_max + k;
  float sum = 0.f;
  for (int c = 0; c < a.g.kc_count; ++c) sum += p[c * a.g.r_max];
  return u.scale * sum;
}

// The y lines of n token rows (rows r0.. of the unit's window), columns
// [col_base, col_base + pcn), into this SM's L1: issued while the current
// tile computes, so the next tile's read-modify-write finds them there
// (one tile at a time; with tiles side by side it measured no better).
// Called after the kernel's wait only (no earlier kernel still writes y).
template <typename TY>
__device__ __forceinline__ void prefetch_rows_l1(const TY *y, int64_t ldy, int col_base, int pcn, const int *rows,
                                                 int r0, int n) {
  const int row_bytes = pcn * (int)sizeof(TY);
  const int lines = (row_bytes + 127) / 128;
  for (int i = threadIdx.x; i < n * lines; i += kThreads) {
    const int t = i / lines, l = i - t * lines;
    const char *p = reinterpret_cast<const char *>(y + (int64_t)rows[(r0 + t) % kRowsWin] * ldy + col_base) + l * 128;
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
  }
}

// The token passes of one expand unit of several tiles: a pass takes NG
// tiles (kTT * NG tokens) at once, tile q of the pass on thread group q of
// kThreads / NG threads; u of a pass is [kTT * NG][r_max] in shared memory,
// zero past the unit.
template <typename TW, typename TY, int NG>
__device__ __forceinline__ void expand_passes(const BgmvArgs &a, const Unit &u, int s, int *rows, float *us,
                                              const TW *Bs, TY *y, int col_base, int pcn, int r_pad) {
  const Geo &g = a.g;
  const int r_max = g.r_max;
  // u of token t (of the unit) and rank index k: the partials summed in chunk
  // order and scaled, or the u buffer. A tile's values go to one of two buffers.
  auto u_val = [&](int tok, int k) -> float {
    if (k >= u.r_a) return 0.f;
    if (a.u_parts) return u_from_partials(a, s, u.start + tok, k, u);
    return a.u_in[((int64_t)s * a.mv.num_tokens + rows[tok % kRowsWin]) * r_max + k];
  };
  constexpr int GS = kThreads / NG;
  const int tpp = kTT * NG;
  const int grp = (int)threadIdx.x / GS, lt = (int)threadIdx.x - grp * GS;
  auto fill = [&](int pass, float *dst) {
    const int n = min(tpp, u.cnt - pass * tpp);
    for (int i = threadIdx.x; i < tpp * r_max; i += kThreads) {
      const int t = i / r_max, k = i - t * r_max;
      dst[i] = t < n ? u_val(pass * tpp + t, k) : 0.f;
    }
  };
  // The next pass's partials are loaded into registers before this pass's
  // products and summed after them, so their latency is hidden.
  const bool overlap = a.u_parts && g.kc_count <= kKCReg && tpp * r_max <= kThreads;
  const int npass = (u.cnt + tpp - 1) / tpp;
  fill(0, us);
  for (int pass = 0; pass < npass; ++pass) {
    float *cur = us + (pass & 1) * tpp * r_max, *nxt_us = us + ((pass + 1) & 1) * tpp * r_max;
    cp_async_wait_upto(0);
    __syncthreads();  // the B chunk, this pass's u and token rows are in shared memory
    const int nxt = pass + 1;
    const bool next_in_window = nxt < npass && (nxt * tpp) % kRowsWin != 0;
    float pref[kKCReg];
    const int i = threadIdx.x, pt = i / r_max, pk = i - pt * r_max;
    const bool mine = overlap && next_in_window && i < tpp * r_max && pt < min(tpp, u.cnt - nxt * tpp) &&
                      pk < u.r_a;
    if (mine) {
      const float *p = a.u_in + (((int64_t)s * a.mv.num_tokens + u.start + nxt * tpp + pt) * g.kc_count) * r_max + pk;
#pragma unroll
      for (int c = 0; c < kKCReg; ++c)
        if (c < g.kc_count) pref[c] = p[c * r_max];
    }
    const int tok0 = pass * tpp + grp * kTT, nt = min(kTT, u.cnt - tok0);
    if (nt > 0)
      expand_pass<TW, TY, GS>(Bs, g.pw, cur + grp * kTT * r_max, r_max, r_pad, rows, tok0, nt, y, a.ldy, col_base,
                              pcn, lt);
    if (nxt < npass) {
      if (!next_in_window) {  // a new window of token rows
        __syncthreads();
        for (int j = threadIdx.x; j < kRowsWin && nxt * tpp + j < u.cnt; j += kThreads)
          rows[j] = a.mv.sorted_rows[u.start + nxt * tpp + j];
        __syncthreads();
        if ((int)threadIdx.x < min(u.cnt - nxt * tpp, kRowsWin))
          prefetch_l2(y + (int64_t)rows[threadIdx.x] * a.ldy + col_base, (uint32_t)(pcn * sizeof(TY)));
        fill(nxt, nxt_us);
      } else if (overlap) {
        if (i < tpp * r_max) {
          float v = 0.f;
          if (mine) {  // same order and arithmetic as u_from_partials
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kKCReg; ++c)
              if (c < g.kc_count) sum += pref[c];
            v = u.scale * sum;
          }
          nxt_us[i] = v;
        }
      } else {
        fill(nxt, nxt_us);
      }
    }
  }
}

// Expand: one CTA per (segment, slice, column chunk of pw). Grid: (chunks over all slices, max_items).
// u comes from the chunk partials (u_parts) or from the u buffer.
template <typename TW, typename TY, bool GROUPS>
__global__ void __launch_bounds__(kThreads, 3) bgmv_expand_kernel(BgmvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  // Behind this library's shrink (or reduce), the metadata and the slot
  // table are complete (see pdl_wait): the record, the B chunk and the y
  // prefetch go out before the wait and overlap the shrink's tail.
  if (!a.pre) {
    pdl_wait();
    pdl_trigger();
  }
  const Geo &g = a.g;
  int s = 0;
  while (s + 1 < a.n_slices && (int)blockIdx.x >= a.chunk_start[s + 1]) ++s;
  int *rows = reinterpret_cast<int *>(smem + g.off_rows);
  Unit u;
  if (!load_unit(a, blockIdx.y, u, smem, rows)) {
    if (a.pre) pdl_wait();
    return;
  }
  const int out_s = a.out_sizes[s];
  const int pc0 = ((int)blockIdx.x - a.chunk_start[s]) * g.pw;
  const int pcn = min(g.pw, out_s - pc0);
  const int r_max = g.r_max;
  const int r_pad = (u.r_a + 1) & ~1;
  TW *Bs = reinterpret_cast<TW *>(smem + g.off_b);
  float *us = reinterpret_cast<float *>(smem + g.off_u);
  const TW *Bslot = static_cast<const TW *>(a.B[s]) + (int64_t)u.slot * r_max * out_s;
  TY *y = static_cast<TY *>(a.y);
  const int col_base = a.out_off[s] + pc0;
  issue_b<TW>(Bs, g.pw, Bslot, out_s, u.r_a, pc0, pcn);
  cp_async_commit();
  if (r_pad > u.r_a)  // odd rank: the partner row of the last pair is zero
    for (int c = threadIdx.x; c < g.pw; c += kThreads) Bs[u.r_a * g.pw + c] = Elem<TW>::from_f(0.f);
  // Token i of the unit is row rows[i % kRowsWin]; the first kTT came with
  // the record, the rest of the window (metadata, complete before this kernel
  // starts behind this library's shrink) and their y lines are fetched now.
  for (int i = kTT + (int)threadIdx.x; i < min(u.cnt, kRowsWin); i += kThreads)
    rows[i] = a.mv.sorted_rows[u.start + i];
  __syncthreads();
  if ((int)threadIdx.x < min(u.cnt, kRowsWin))
    prefetch_l2(y + (int64_t)rows[threadIdx.x] * a.ldy + col_base, (uint32_t)(pcn * sizeof(TY)));
  if (a.pre) {
    pdl_wait();
    pdl_trigger();
  }
  // A chunk narrower than half the block's reach (4 columns per thread)
  // would leave threads idle (GROUPS), so a unit of several tiles runs up to
  // that many tiles at once, tile q of a pass on thread group q. Every output
  // takes the same arithmetic for any group count. Wider chunks keep one tile
  // at a time: there, running tiles side by side measured slower.
  if constexpr (GROUPS) {
    const int ng_geo = g.pw * 4 <= kReach ? 4 : 2;
    const int nt_all = (u.cnt + kTT - 1) / kTT;
    const int ng = min(ng_geo, nt_all >= 3 ? 4 : nt_all);
    if (ng == 4) return expand_passes<TW, TY, 4>(a, u, s, rows, us, Bs, y, col_base, pcn, r_pad);
    if (ng == 2) return expand_passes<TW, TY, 2>(a, u, s, rows, us, Bs, y, col_base, pcn, r_pad);
  }
  // One tile at a time. u of token t (of the unit) and rank index k: the partials summed in chunk
  // order and scaled, or the u buffer. A tile's values go to one of two buffers.
  auto u_val = [&](int tok, int k) -> float {
    if (k >= u.r_a) return 0.f;
    if (a.u_parts) return u_from_partials(a, s, u.start + tok, k, u);
    return a.u_in[((int64_t)s * a.mv.num_tokens + rows[tok % kRowsWin]) * r_max + k];
  };
  auto fill = [&](int tile, float *dst) {
    const int nt = min(kTT, u.cnt - tile * kTT);
    for (int i = threadIdx.x; i < kTT * r_max; i += kThreads) {
      const int t = i / r_max, k = i - t * r_max;
      dst[i] = t < nt ? u_val(tile * kTT + t, k) : 0.f;
    }
  };
  // The next tile's partials are loaded into registers before this tile's
  // products and summed after them, so their latency is hidden.
  const bool overlap = a.u_parts && g.kc_count <= kKCReg && kTT * r_max <= kThreads;
  const int ntiles = (u.cnt + kTT - 1) / kTT;
  fill(0, us);
  for (int tile = 0; tile < ntiles; ++tile) {
    const int nt = min(kTT, u.cnt - tile * kTT);
    float *cur = us + (tile & 1) * kTT * r_max, *nxt_us = us + ((tile + 1) & 1) * kTT * r_max;
    cp_async_wait_upto(0);
    __syncthreads();  // the B chunk, this tile's u and token rows are in shared memory
    const int nxt = tile + 1;
    const bool next_in_window = nxt < ntiles && (nxt * kTT) % kRowsWin != 0;
    float pref[kKCReg];
    const int i = threadIdx.x, pt = i / r_max, pk = i - pt * r_max;
    const bool mine = overlap && next_in_window && i < kTT * r_max && pt < min(kTT, u.cnt - nxt * kTT) &&
                      pk < u.r_a;
    if (mine) {
      const float *p = a.u_in + (((int64_t)s * a.mv.num_tokens + u.start + nxt * kTT + pt) * g.kc_count) * r_max + pk;
#pragma unroll
      for (int c = 0; c < kKCReg; ++c)
        if (c < g.kc_count) pref[c] = p[c * r_max];
    }
    if (next_in_window) prefetch_rows_l1(y, a.ldy, col_base, pcn, rows, nxt * kTT, min(kTT, u.cnt - nxt * kTT));
    expand_pass<TW, TY, kThreads>(Bs, g.pw, cur, r_max, r_pad, rows, tile * kTT, nt, y, a.ldy, col_base,
                                    pcn, (int)threadIdx.x);
    if (nxt < ntiles) {
      if (!next_in_window) {  // a new window of token rows
        __syncthreads();
        for (int j = threadIdx.x; j < kRowsWin && nxt * kTT + j < u.cnt; j += kThreads)
          rows[j] = a.mv.sorted_rows[u.start + nxt * kTT + j];
        __syncthreads();
        if ((int)threadIdx.x < min(u.cnt - nxt * kTT, kRowsWin))
          prefetch_l2(y + (int64_t)rows[threadIdx.x] * a.ldy + col_base, (uint32_t)(pcn * sizeof(TY)));
        fill(nxt, nxt_us);
      } else if (overlap) {
        if (i < kTT * r_max) {
          float v = 0.f;
          if (mine) {  // same order and arithmetic as u_from_partials
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kKCReg; ++c)
              if (c < g.kc_count) sum += pref[c];
            v = u.scale * sum;
          }
          nxt_us[i] = v;
        }
      } else {
        fill(nxt, nxt_us);
      }
    }
  }
}

// ------------------------------------------------------------------ launchers (one translation unit each)

cudaError_t dispatch_shrink_bf16(const BgmvArgs &a, cudaStream_t st);
cudaError_t dispatch_shrink_f32(const BgmvArgs &a, cudaStream_t st);
cudaError_t launch_expand(const BgmvArgs &a, int dtype, int y_dtype, cudaStream_t st);
cudaError_t launch_reduce(const BgmvArgs &a, cudaStream_t st);

}  // namespace bgmvk
}  // namespace ra
