// BGMV shrink / expand on CUDA cores: the decode form of the multi-LoRA delta
// (handbook page "多 LoRA 服务：分段矩阵乘与适配器调度", section "不合并权重，批量计算":
// each token gathers its own adapter and does a small matrix-vector product).
//
// Decode is bound by reading each active adapter's A and B once from HBM
// (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section "成本与边界": about
// 2 r (d_in + d_out) extra elements per layer), so the kernels are organised
// around the weights. A work unit is one (segment, slice).
//
// * shrink / apply: a persistent grid of thread-block clusters, as many as
//   fit resident. Cluster c walks units c, c + NC, ...; its CS CTAs split
//   d_in. Each CTA runs a two-stage pipeline: while it computes one unit,
//   the next unit's A rows, x rows and (fused) B columns are already in
//   flight through 16-byte cp.async copies, and its y rows are being pulled
//   into L2. A thread widens a 16-byte weight vector once and applies it to
//   the 4 tokens of a tile held in registers; row groups combine by a
//   recursive-halving shuffle reduce-scatter and a fixed-order sum over
//   warps; the CS CTA partials meet in distributed shared memory, summed in
//   cluster-rank order (deterministic split-K: no global scratch, no atomics,
//   no spin waits). The fused kernel then adds u B into each CTA's share of
//   the slice's columns; results are bitwise those of shrink then expand.
// * expand: one CTA per (segment, slice, column chunk).
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTT = 4;                 // tokens per tile
constexpr int kAStageBytes = 32768;    // A bytes of one pipeline buffer (longer K shares go in stretches)
constexpr int kBPassBytes = 32768;     // B bytes staged per pass
constexpr int kSmallTable = 256;       // slot tables up to this size: rank / scale copied whole

struct Geo {
  int d_in, r_max, kc;   // kc: d_in rows per cluster CTA
  int sc_rows;           // A rows per pipeline buffer
  int pw;                // B columns per pass
  int off_a, off_x, off_red, off_cpart, off_u, off_rows, off_b, off_rs, off_rec, smem;
  int a_stage, x_stage, b_stage;   // bytes of one pipeline buffer of each kind
};

struct BgmvArgs {
  const void *x;
  int64_t ldx;
  const void *A[LORA_MAX_SLICES];
  const void *B[LORA_MAX_SLICES];
  float *buf;  // may be null for the fused kernel
  void *y;
  int64_t ldy;
  int out_sizes[LORA_MAX_SLICES];
  int out_off[LORA_MAX_SLICES];
  MetaView mv;
  int list;      // int offset of the unit-record list inside the work lists
  int list_cnt;  // header index of that list's length
  int n_slices;
  const int32_t *slot_rank;
  const float *slot_scale;
  Geo g;
};

struct Unit {
  int slot, cnt, start, r_a;
  float scale;
};

// One unit record (segment, slot, count, start, first rows) and the slot's
// rank and scale. Small slot tables are copied whole into shared memory in
// parallel with the record, so everything arrives in one round trip.
// The record's first rows go to rows[0..kTT). Returns false (uniformly over
// the CTA and its cluster) for an unused record.
__device__ __forceinline__ bool load_unit(const BgmvArgs &a, int item, Unit &u, int32_t *rank_s, float *scale_s,
                                          int *rows) {
  const int S = a.mv.num_slots;
  const bool small_table = S <= kSmallTable;
  if (small_table) {
    for (int i = threadIdx.x; i < S; i += kThreads) {
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

// 16 bytes of weights widened to fp32.
template <typename TW>
__device__ __forceinline__ void widen16(const uint4 &q, float *f) {
  if constexpr (sizeof(TW) == 2) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
  }
}

// 4 consecutive elements of a row, widened (8 bytes of bf16 or 16 of fp32).
template <typename T>
__device__ __forceinline__ void load4(const T *p, float *f) {
  if constexpr (sizeof(T) == 2) {
    const uint2 q = *reinterpret_cast<const uint2 *>(p);
    f[0] = __uint_as_float(q.x << 16); f[1] = __uint_as_float(q.x & 0xffff0000u);
    f[2] = __uint_as_float(q.y << 16); f[3] = __uint_as_float(q.y & 0xffff0000u);
  } else {
    const float4 q = *reinterpret_cast<const float4 *>(p);
    f[0] = q.x; f[1] = q.y; f[2] = q.z; f[3] = q.w;
  }
}
template <typename T>
__device__ __forceinline__ void store4(T *p, const float *f) {
  if constexpr (sizeof(T) == 2) {
    uint2 q;
    __nv_bfloat162 lo = __floats2bfloat162_rn(f[0], f[1]), hi = __floats2bfloat162_rn(f[2], f[3]);
    q.x = *reinterpret_cast<uint32_t *>(&lo);
    q.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = q;
  } else {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
}

// Sum N values per lane over the lanes that share bits [0, log2(NV)) of the
// lane id (recursive halving). Afterwards lane keeps N / (32 / NV) sums in
// vals[0..) whose positions in the original array start at the returned offset.
template <int N, int NV>
__device__ __forceinline__ int reduce_scatter(float (&vals)[N]) {
  const int lane = threadIdx.x & 31;
  int off = 0;
#pragma unroll
  for (int lvl = 0, o = NV; o < 32; ++lvl, o <<= 1) {
    const int cnt = N >> lvl;
    const int half = cnt >> 1;
    if (half == 0) break;
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

// Add u . B into y for tokens [0, nt) over columns [pc0, pc0 + pcn) of a
// slice. Bs: B rows 0..r_a-1 of those columns (row stride pw); uT: u
// transposed, [r_max][kTT]. One thread per 4 columns, all tokens of the tile.
template <typename TW, typename TY>
__device__ __forceinline__ void expand_pass(const TW *Bs, int pw, const float *uT, int r_a, const int *rows,
                                            int nt, TY *y, int64_t ldy, int col_base, int pcn) {
  for (int cq = threadIdx.x * 4; cq < pcn; cq += kThreads * 4) {
    float acc[kTT][4];
#pragma unroll
    for (int t = 0; t < kTT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
    const TW *bp = Bs + cq;
#pragma unroll 4
    for (int k = 0; k < r_a; ++k) {
      float b[4];
      load4(bp + k * pw, b);
      const float4 u4 = *reinterpret_cast<const float4 *>(uT + k * kTT);
      const float uu[kTT] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int t = 0; t < kTT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = fmaf(uu[t], b[e], acc[t][e]);
    }
#pragma unroll
    for (int t = 0; t < kTT; ++t) {
      if (t < nt) {
        TY *yp = y + (int64_t)rows[t] * ldy + col_base + cq;
        float yv[4];
        load4(yp, yv);
#pragma unroll
        for (int e = 0; e < 4; ++e) yv[e] += acc[t][e];
        store4(yp, yv);
      }
    }
  }
}

// B rows 0..r_a-1, columns [pc0, pc0 + pcn) of one slot -> Bs (row stride pw). A warp per row.
template <typename TW>
__device__ __forceinline__ void issue_b(TW *Bs, int pw, const TW *Bslot, int out_s, int r_a, int pc0, int pcn) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int upr = pcn * (int)sizeof(TW) / 16;
  for (int k = warp; k < r_a; k += kWarps) {
    const char *src = reinterpret_cast<const char *>(Bslot + (int64_t)k * out_s + pc0);
    char *dst = reinterpret_cast<char *>(Bs + k * pw);
    for (int c = lane; c < upr; c += 32) cp_async16(dst + c * 16, src + c * 16);
  }
}

// Everything a CTA needs about one unit, resolved from the staged records.
struct UnitInfo {
  int slice, slot, cnt, start, r_a;
  float scale;
  int4 rows;   // first 4 token rows of the segment (-1 past the count)
};

// Shrink (kApply = false) or fused shrink + expand (kApply = true).
// Grid: NC * CS CTAs in clusters of CS, all resident; see the file comment.
template <typename TW, typename TY, int NV, bool kApply>
__global__ void __launch_bounds__(kThreads, 2) bgmv_kernel(BgmvArgs a) {
  constexpr int VEC = Elem<TW>::kVec;
  constexpr int NRG = kThreads / NV;   // row groups
  constexpr int NVAL = kTT * VEC;      // accumulators per thread
  constexpr int LPV = 32 / NV;         // lanes sharing one vector column
  constexpr int NKEEP = NVAL / (LPV > NVAL ? NVAL : LPV);
  constexpr int kMaxCS = 8;
  extern __shared__ __align__(16) unsigned char smem[];
  const Geo &g = a.g;
  const int cs = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
  const int cid = blockIdx.x / cs, ncl = gridDim.x / cs;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int v = tid % NV, rq = tid / NV;
  const int S = a.mv.num_slots, r_max = g.r_max;
  const bool small_table = S <= kSmallTable;
  const int32_t *W = a.mv.work;
  int4 *rec_s = reinterpret_cast<int4 *>(smem + g.off_rec);        // [min(S, kSmallTable)] records
  int32_t *rank_s = reinterpret_cast<int32_t *>(smem + g.off_rs);  // [kSmallTable]
  float *scale_s = reinterpret_cast<float *>(rank_s + kSmallTable);
  int *rows_s = reinterpret_cast<int *>(smem + g.off_rows);        // [2][kTT] rows of the buffered tile
  float *wred = reinterpret_cast<float *>(smem + g.off_red);       // [kWarps][kTT][r_max]
  float *cpart = reinterpret_cast<float *>(smem + g.off_cpart);    // [kTT][r_max]
  float *uT = reinterpret_cast<float *>(smem + g.off_u);           // [r_max][kTT]
  __shared__ int n_list_s;

  // One round trip: list length, unit records, slot ranks and scales.
  const int nrec = min(S, kSmallTable);
  for (int i = tid; i < 2 * nrec; i += kThreads)
    cp_async16(rec_s + i, W + a.list + 4 * i);
  if (small_table) {
    for (int i = tid; i < S; i += kThreads) {
      rank_s[i] = a.slot_rank[i];
      scale_s[i] = a.slot_scale[i];
    }
  }
  if (tid == 0) n_list_s = W[a.list_cnt];
  cp_async_commit();
  cp_async_wait_upto(0);
  __syncthreads();
  const int n_units = n_list_s * a.n_slices;
  const TW *x = static_cast<const TW *>(a.x);
  TY *y = static_cast<TY *>(a.y);
  const int j0 = crank * g.kc;
  const int len = max(0, min(g.d_in - j0, g.kc));

  auto info = [&](int u, UnitInfo &ui) {
    const int item = u / a.n_slices;
    ui.slice = u - item * a.n_slices;
    int4 h, r;
    if (item < nrec) {
      h = rec_s[2 * item];
      r = rec_s[2 * item + 1];
    } else {
      h = *reinterpret_cast<const int4 *>(W + a.list + item * WorkLists::kRec);
      r = *reinterpret_cast<const int4 *>(W + a.list + item * WorkLists::kRec + 4);
    }
    ui.slot = h.y;
    ui.cnt = h.z;
    ui.start = h.w;
    ui.rows = r;
    const int rk = small_table ? rank_s[ui.slot] : a.slot_rank[ui.slot];
    ui.r_a = min(max(rk, 0), r_max);
    ui.scale = small_table ? scale_s[ui.slot] : a.slot_scale[ui.slot];
  };
  // Columns of the slice this CTA adds into (fused kernel).
  auto cols = [&](const UnitInfo &ui, int &c0, int &c1) {
    const int out_s = a.out_sizes[ui.slice];
    const int per = ((out_s + cs - 1) / cs + 7) & ~7;
    c0 = min(out_s, crank * per);
    c1 = min(out_s, c0 + per);
  };
  auto bufA = [&](int b) { return reinterpret_cast<TW *>(smem + g.off_a + b * g.a_stage); };
  auto bufX = [&](int b) { return reinterpret_cast<TW *>(smem + g.off_x + b * g.x_stage); };
  auto bufB = [&](int b) { return reinterpret_cast<TW *>(smem + g.off_b + b * g.b_stage); };

  // Put x rows of tokens [0, nt) (rows in rows_s[b]) into buffer b; a warp per row.
  auto issue_x = [&](int b, int nt) {
    const int upr = len / VEC;
    TW *xs = bufX(b);
    for (int t = warp; t < nt; t += kWarps) {
      const TW *src = x + (int64_t)rows_s[b * kTT + t] * a.ldx + j0;
      for (int c = tid & 31; c < upr; c += 32) cp_async16(xs + t * g.kc + c * VEC, src + c * VEC);
    }
  };
  // A rows [j0 + r0, j0 + r0 + nr) of the unit's slot into buffer b: one flat copy, rank tail skipped.
  auto issue_rows = [&](const UnitInfo &ui, int b, int r0, int nr, int nva) {
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const TW *>(a.A[ui.slice]) +
                                                       ((int64_t)ui.slot * g.d_in + j0 + r0) * r_max);
    uint4 *dst = reinterpret_cast<uint4 *>(bufA(b));
    for (int i = tid; i < nr * NV; i += kThreads)
      if ((i & (NV - 1)) < nva) cp_async16(dst + i, src + i);
  };
  const int nsc = (len + g.sc_rows - 1) / g.sc_rows;
  // Stage unit u into buffer b: A rows, x rows and B columns of the first tile; y rows to L2.
  int committed = 0;
  int g_buf0 = -1, g_buf1 = -1;   // commit group of each buffer's staged unit
  auto stage = [&](int u, int b) {
    UnitInfo ui;
    info(u, ui);
    const int nt = min(kTT, ui.cnt);
    if (tid < kTT) {
      const int rv = tid == 0 ? ui.rows.x : tid == 1 ? ui.rows.y : tid == 2 ? ui.rows.z : ui.rows.w;
      rows_s[b * kTT + tid] = rv;
    }
    issue_rows(ui, b, 0, min(g.sc_rows, len), (ui.r_a + VEC - 1) / VEC);
    {  // x rows of the first tile; row ids straight from the record
      const int upr = len / VEC;
      TW *xs = bufX(b);
      for (int t = warp; t < nt; t += kWarps) {
        const int row = t == 0 ? ui.rows.x : t == 1 ? ui.rows.y : t == 2 ? ui.rows.z : ui.rows.w;
        const TW *xsrc = x + (int64_t)row * a.ldx + j0;
        for (int c = tid & 31; c < upr; c += 32) cp_async16(xs + t * g.kc + c * VEC, xsrc + c * VEC);
      }
    }
    if constexpr (kApply) {
      int c0, c1;
      cols(ui, c0, c1);
      if (c1 > c0) {
        const int out_s = a.out_sizes[ui.slice];
        const TW *Bslot = static_cast<const TW *>(a.B[ui.slice]) + (int64_t)ui.slot * r_max * out_s;
        issue_b<TW>(bufB(b), g.pw, Bslot, out_s, ui.r_a, c0, min(g.pw, c1 - c0));
        if (tid < nt) {
          const int row = tid == 0 ? ui.rows.x : tid == 1 ? ui.rows.y : tid == 2 ? ui.rows.z : ui.rows.w;
          prefetch_l2(y + (int64_t)row * a.ldy + a.out_off[ui.slice] + c0, (uint32_t)((c1 - c0) * sizeof(TY)));
        }
      }
    }
    cp_async_commit();
    if (b) g_buf1 = committed++; else g_buf0 = committed++;
  };

  int u0 = cid;
  if (u0 < n_units) stage(u0, 0);
  if (u0 + ncl < n_units) stage(u0 + ncl, 1);
  for (int k = 0, u = u0; u < n_units; ++k, u += ncl) {
    const int b = k & 1;
    UnitInfo ui;
    info(u, ui);
    const int nva = (ui.r_a + VEC - 1) / VEC;
    cp_async_wait_upto(committed - 1 - (b ? g_buf1 : g_buf0));
    __syncthreads();
    const TW *As = bufA(b) + v * VEC;
    const TW *xs = bufX(b);
    int c0 = 0, c1 = 0;
    if (kApply) cols(ui, c0, c1);
    const int npass = (c1 - c0 + g.pw - 1) / g.pw;
    const int out_s = a.out_sizes[ui.slice];
    const TW *Bslot = static_cast<const TW *>(a.B[ui.slice]) + (int64_t)ui.slot * r_max * out_s;
    const int ntiles = (ui.cnt + kTT - 1) / kTT;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int nt = min(kTT, ui.cnt - tile * kTT);
      if (tile > 0) {  // later tiles of a long segment: fetch rows and x synchronously
        __syncthreads();
        if (tid < nt) rows_s[b * kTT + tid] = a.mv.sorted_rows[ui.start + tile * kTT + tid];
        __syncthreads();
        issue_x(b, nt);
        cp_async_commit();
        ++committed;
        cp_async_wait_upto(0);
        __syncthreads();
      }
      float acc[NVAL];
#pragma unroll
      for (int i = 0; i < NVAL; ++i) acc[i] = 0.f;
      for (int sc = 0; sc < nsc; ++sc) {
        const int r0 = sc * g.sc_rows, nr = min(g.sc_rows, len - r0);
        if (sc > 0 || (tile > 0 && nsc > 1)) {  // this stretch of A is not resident: load it now
          __syncthreads();
          issue_rows(ui, b, r0, nr, nva);
          cp_async_commit();
          ++committed;
          cp_async_wait_upto(0);
          __syncthreads();
        }
        if (v < nva) {
          const TW *xr = xs + r0;
#pragma unroll 2
          for (int jj = rq; jj < nr; jj += NRG) {
            float af[VEC];
            widen16<TW>(*reinterpret_cast<const uint4 *>(As + jj * r_max), af);
            float xv[kTT];
#pragma unroll
            for (int t = 0; t < kTT; ++t) xv[t] = Elem<TW>::to_f(xr[t * g.kc + jj]);
#pragma unroll
            for (int t = 0; t < kTT; ++t)
#pragma unroll
              for (int e = 0; e < VEC; ++e) acc[t * VEC + e] = fmaf(xv[t], af[e], acc[t * VEC + e]);
          }
        }
      }
      // Row groups inside a warp, warps in order, then cluster CTAs in rank order.
      // Entries of absent tokens (t >= nt) carry garbage and are never used.
      const int off = reduce_scatter<NVAL, NV>(acc);
#pragma unroll
      for (int i = 0; i < NKEEP; ++i) {
        const int idx = off + i, t = idx / VEC, e = idx % VEC;
        wred[(warp * kTT + t) * r_max + v * VEC + e] = acc[i];
      }
      __syncthreads();
      for (int i = tid; i < nt * r_max; i += kThreads) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += wred[w * kTT * r_max + i];
        cpart[i] = sum;
      }
      cluster_sync();
      if (kApply || crank == 0) {
        const int r4 = r_max >> 2;
        for (int i = tid; i < nt * r4; i += kThreads) {
          const int tt = i / r4, kk = (i - tt * r4) * 4;
          const uint32_t la = smem_addr(cpart + tt * r_max + kk);
          float4 p[kMaxCS];
#pragma unroll
          for (int c = 0; c < kMaxCS; ++c)
            if (c < cs) p[c] = ld_dsmem_f4(la, (uint32_t)c);
          float4 sm = p[0];
#pragma unroll
          for (int c = 1; c < kMaxCS; ++c)
            if (c < cs) { sm.x += p[c].x; sm.y += p[c].y; sm.z += p[c].z; sm.w += p[c].w; }
          const float o[4] = {(kk + 0 < ui.r_a) ? ui.scale * sm.x : 0.f, (kk + 1 < ui.r_a) ? ui.scale * sm.y : 0.f,
                              (kk + 2 < ui.r_a) ? ui.scale * sm.z : 0.f, (kk + 3 < ui.r_a) ? ui.scale * sm.w : 0.f};
          if (kApply) {
#pragma unroll
            for (int e = 0; e < 4; ++e) uT[(kk + e) * kTT + tt] = o[e];
          }
          if (crank == 0 && a.buf != nullptr)
            *reinterpret_cast<float4 *>(a.buf + ((int64_t)ui.slice * a.mv.num_tokens + rows_s[b * kTT + tt]) * r_max +
                                        kk) = make_float4(o[0], o[1], o[2], o[3]);
        }
        if (kApply) {  // absent tokens of the tile contribute nothing
          for (int i = tid; i < (kTT - nt) * r_max; i += kThreads) {
            const int tt = nt + i / r_max, kk = i % r_max;
            uT[kk * kTT + tt] = 0.f;
          }
        }
      }
      cluster_sync();  // partials read; cpart may be rewritten, peers may move on
      if constexpr (kApply) {
        for (int pass = 0; pass < npass; ++pass) {
          const int pc0 = c0 + pass * g.pw, pcn = min(g.pw, c1 - pc0);
          const bool resident = (pass == 0 && tile == 0) || (npass == 1 && tile > 0);
          if (!resident) {
            __syncthreads();
            issue_b<TW>(bufB(b), g.pw, Bslot, out_s, ui.r_a, pc0, pcn);
            cp_async_commit();
            ++committed;
            cp_async_wait_upto(0);
          }
          __syncthreads();
          expand_pass<TW, TY>(bufB(b), g.pw, uT, ui.r_a, rows_s + b * kTT, nt, y, a.ldy,
                              a.out_off[ui.slice] + pc0, pcn);
        }
      }
    }
    __syncthreads();  // buffer b is free: stage the unit after next into it
    if (u + 2 * ncl < n_units) stage(u + 2 * ncl, b);
  }
  cp_async_wait_upto(0);
}

// Standalone expand. Grid: (column chunks over all slices, max_items).
struct ExpandArgs {
  BgmvArgs b;
  int chunk_start[LORA_MAX_SLICES + 1];
  int n_slices;
};

template <typename TW, typename TY>
__global__ void __launch_bounds__(kThreads, 4) bgmv_expand_kernel(ExpandArgs ea) {
  const BgmvArgs &a = ea.b;
  const Geo &g = a.g;
  extern __shared__ __align__(16) unsigned char smem[];
  TW *Bs = reinterpret_cast<TW *>(smem + g.off_b);
  float *uT = reinterpret_cast<float *>(smem + g.off_u);
  int *rows = reinterpret_cast<int *>(smem + g.off_rows);
  int32_t *rank_s = reinterpret_cast<int32_t *>(smem + g.off_rs);
  float *scale_s = reinterpret_cast<float *>(rank_s + kSmallTable);
  Unit u;
  if (!load_unit(a, blockIdx.y, u, rank_s, scale_s, rows)) return;
  int s = 0;
  while (s + 1 < ea.n_slices && (int)blockIdx.x >= ea.chunk_start[s + 1]) ++s;
  const int out_s = a.out_sizes[s];
  const int pc0 = ((int)blockIdx.x - ea.chunk_start[s]) * g.pw;
  const int pcn = min(g.pw, out_s - pc0);
  const int r_max = g.r_max;
  const TW *Bslot = static_cast<const TW *>(a.B[s]) + (int64_t)u.slot * r_max * out_s;
  const float *bufs = a.buf + (int64_t)s * a.mv.num_tokens * r_max;
  TY *y = static_cast<TY *>(a.y);
  const int col_base = a.out_off[s] + pc0;
  issue_b<TW>(Bs, g.pw, Bslot, out_s, u.r_a, pc0, pcn);
  cp_async_commit();
  const int ntiles = (u.cnt + kTT - 1) / kTT;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int tok0 = tile * kTT, nt = min(kTT, u.cnt - tok0);
    if (tile > 0) {
      __syncthreads();
      if (threadIdx.x < nt) rows[threadIdx.x] = a.mv.sorted_rows[u.start + tok0 + threadIdx.x];
      __syncthreads();
    }
    if (threadIdx.x < nt) prefetch_l2(y + (int64_t)rows[threadIdx.x] * a.ldy + col_base, (uint32_t)(pcn * sizeof(TY)));
    for (int i = threadIdx.x; i < kTT * r_max; i += kThreads) {
      const int tt = i / r_max, k = i - tt * r_max;
      uT[k * kTT + tt] = (tt < nt && k < u.r_a) ? bufs[(int64_t)rows[tt] * r_max + k] : 0.f;
    }
    cp_async_wait_upto(0);
    __syncthreads();
    expand_pass<TW, TY>(Bs, g.pw, uT, u.r_a, rows, nt, y, a.ldy, col_base, pcn);
  }
}

int align16(int v) { return (v + 15) & ~15; }

int cluster_size(int d_in) {
  int cs = d_in / 512;
  return cs < 1 ? 1 : (cs > 8 ? 8 : cs);
}

// Shared-memory geometry. mode: 0 shrink, 1 expand, 2 fused apply.
// Shrink / apply hold two pipeline buffers of each kind; the standalone
// expand holds one B chunk.
Geo make_geo(const lora_layer_desc &d, int cs, int mode) {
  Geo g{};
  const int es = d.dtype == LORA_BF16 ? 2 : 4;
  g.d_in = d.d_in;
  g.r_max = d.r_max;
  g.kc = (((d.d_in + cs - 1) / cs) + 7) & ~7;
  const int row_bytes = d.r_max * es;
  g.sc_rows = g.kc * row_bytes <= kAStageBytes ? g.kc : ((kAStageBytes / row_bytes) & ~7);
  if (g.sc_rows < 8) g.sc_rows = 8;
  int pw = (kBPassBytes / row_bytes) & ~7;
  if (pw < 8) pw = 8;
  int max_cols = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    const int per = mode == 2 ? ((((d.out_sizes[s] + cs - 1) / cs) + 7) & ~7) : d.out_sizes[s];
    max_cols = per > max_cols ? per : max_cols;
  }
  if (pw > max_cols) pw = max_cols;
  g.pw = pw;
  const int nbuf = mode == 1 ? 1 : 2;
  g.a_stage = mode == 1 ? 0 : align16(g.sc_rows * row_bytes);
  g.x_stage = mode == 1 ? 0 : align16(kTT * g.kc * es);
  g.b_stage = mode == 0 ? 0 : align16(d.r_max * pw * es);
  int off = 0;
  g.off_rs = off;
  off += align16(2 * kSmallTable * 4);
  g.off_rec = off;
  off += align16(kSmallTable * WorkLists::kRec * 4);
  g.off_a = off;
  off += nbuf * g.a_stage;
  g.off_x = off;
  off += nbuf * g.x_stage;
  g.off_b = off;
  off += nbuf * g.b_stage;
  g.off_red = off;
  if (mode != 1) off += align16(kWarps * kTT * d.r_max * 4);
  g.off_cpart = off;
  if (mode != 1) off += align16(kTT * d.r_max * 4);
  g.off_u = off;
  off += align16(kTT * d.r_max * 4);
  g.off_rows = off;
  off += align16(2 * kTT * 4);
  g.smem = off;
  return g;
}

void fill_common(BgmvArgs &a, const lora_layer_desc &d, const MetaView &mv, ListSel sel) {
  a.list = WorkLists::list(mv.num_slots, sel);
  a.list_cnt = sel == kListSmall ? 1 : sel == kListLarge ? 2 : 0;
  a.n_slices = d.n_slices;
  a.mv = mv;
  int off = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    a.A[s] = d.A[s];
    a.B[s] = d.B[s];
    a.out_sizes[s] = d.out_sizes[s];
    a.out_off[s] = off;
    off += d.out_sizes[s];
  }
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
}

// Clusters of `cs` CTAs of kernel k with `smem` bytes that fit resident at once on this device.
int resident_clusters(const void *k, int cs, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, int, int>, int> memo;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const auto key = std::make_tuple(k, cs, smem, dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms / cs > 0 ? sms / cs : 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = n;
  return n;
}

template <typename TW, typename TY, bool kApply, int NV>
cudaError_t launch_nv(const BgmvArgs &a, int cs, int max_units, cudaStream_t st) {
  auto k = bgmv_kernel<TW, TY, NV, kApply>;
  cudaError_t e = set_max_dynamic_smem((const void *)k, a.g.smem);
  if (e != cudaSuccess) return e;
  int ncl = resident_clusters((const void *)k, cs, a.g.smem);
  if (ncl > max_units) ncl = max_units;
  return launch_cluster(k, dim3((unsigned)(ncl * cs)), dim3(kThreads), (size_t)a.g.smem, st, (unsigned)cs, a);
}

template <typename TW, typename TY, bool kApply>
cudaError_t dispatch_nv(BgmvArgs &a, int cs, int max_units, int r_max, cudaStream_t st) {
  const int nv = r_max / Elem<TW>::kVec;
  if constexpr (sizeof(TW) == 2) {
    switch (nv) {
      case 1: return launch_nv<TW, TY, kApply, 1>(a, cs, max_units, st);
      case 2: return launch_nv<TW, TY, kApply, 2>(a, cs, max_units, st);
      case 4: return launch_nv<TW, TY, kApply, 4>(a, cs, max_units, st);
      case 8: return launch_nv<TW, TY, kApply, 8>(a, cs, max_units, st);
      case 16: return launch_nv<TW, TY, kApply, 16>(a, cs, max_units, st);
    }
  } else {
    switch (nv) {
      case 2: return launch_nv<TW, TY, kApply, 2>(a, cs, max_units, st);
      case 4: return launch_nv<TW, TY, kApply, 4>(a, cs, max_units, st);
      case 8: return launch_nv<TW, TY, kApply, 8>(a, cs, max_units, st);
      case 16: return launch_nv<TW, TY, kApply, 16>(a, cs, max_units, st);
      case 32: return launch_nv<TW, TY, kApply, 32>(a, cs, max_units, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_bgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel,
                               const void *x, int64_t ldx, float *buf, cudaStream_t st) {
  const int max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  if (max_items <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.x = x;
  a.ldx = ldx;
  a.buf = buf;
  const int cs = cluster_size(d.d_in);
  a.g = make_geo(d, cs, 0);
  const int max_units = max_items * d.n_slices;
  if (d.dtype == LORA_BF16) return dispatch_nv<__nv_bfloat16, float, false>(a, cs, max_units, d.r_max, st);
  return dispatch_nv<float, float, false>(a, cs, max_units, d.r_max, st);
}

cudaError_t launch_bgmv_apply(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                              int64_t ldx, float *buf, void *y, int64_t ldy, int y_dtype, cudaStream_t st) {
  const int max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  if (max_items <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.x = x;
  a.ldx = ldx;
  a.buf = buf;
  a.y = y;
  a.ldy = ldy;
  const int cs = cluster_size(d.d_in);
  a.g = make_geo(d, cs, 2);
  const int max_units = max_items * d.n_slices;
  if (d.dtype == LORA_BF16) {
    if (y_dtype == LORA_BF16) return dispatch_nv<__nv_bfloat16, __nv_bfloat16, true>(a, cs, max_units, d.r_max, st);
    return dispatch_nv<__nv_bfloat16, float, true>(a, cs, max_units, d.r_max, st);
  }
  return dispatch_nv<float, float, true>(a, cs, max_units, d.r_max, st);
}

cudaError_t launch_bgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel,
                               const float *buf, void *y, int64_t ldy, int y_dtype, cudaStream_t st) {
  const int max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  if (max_items <= 0) return cudaSuccess;
  ExpandArgs ea{};
  BgmvArgs &a = ea.b;
  fill_common(a, d, mv, sel);
  a.buf = const_cast<float *>(buf);
  a.y = y;
  a.ldy = ldy;
  a.g = make_geo(d, 1, 1);
  int chunks = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    ea.chunk_start[s] = chunks;
    chunks += (d.out_sizes[s] + a.g.pw - 1) / a.g.pw;
  }
  ea.chunk_start[d.n_slices] = chunks;
  ea.n_slices = d.n_slices;
  dim3 grid((unsigned)chunks, (unsigned)max_items);
  const size_t smem = (size_t)a.g.smem;
  void (*k)(ExpandArgs);
  if (d.dtype == LORA_BF16 && y_dtype == LORA_BF16) k = bgmv_expand_kernel<__nv_bfloat16, __nv_bfloat16>;
  else if (d.dtype == LORA_BF16) k = bgmv_expand_kernel<__nv_bfloat16, float>;
  else k = bgmv_expand_kernel<float, float>;
  cudaError_t e = set_max_dynamic_smem((const void *)k, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, st>>>(ea);
  return cudaGetLastError();
}

}  // namespace ra
