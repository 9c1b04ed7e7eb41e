// BGMV shrink / expand on CUDA cores: the decode form of the multi-LoRA delta
// (handbook page "多 LoRA 服务：分段矩阵乘与适配器调度", section "不合并权重，批量计算":
// each token gathers its own adapter and does a small matrix-vector product).
//
// Decode is bound by reading each active adapter's A and B once from HBM
// (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section "成本与边界": the extra
// access per layer is about 2 r (d_in + d_out) elements). So the kernels are
// organised around the weights, not the tokens: work units are (segment,
// slice, chunk of the weight matrix), every unit streams its chunk once with
// 16-byte loads, and applies it to all tokens of its segment.
//
// Shrink: a cluster of CS CTAs splits d_in into CS chunks; each CTA reduces
// its chunk with warp shuffles, and CTA 0 sums the CS partials over
// distributed shared memory in a fixed order (deterministic split-K without
// global scratch, atomics or spin waits).
// Expand: one CTA per (segment, slice, 1024-column chunk) reads its B chunk
// once and adds buf . B into the token rows of y.
#include "common.cuh"

namespace ra {
namespace {

constexpr int kTT = 8;              // tokens per tile
constexpr int kShrinkThreads = 256;
constexpr int kShrinkWarps = kShrinkThreads / 32;
constexpr int kExpandThreads = 128;
constexpr int kExpandCols = kExpandThreads * 8;

struct ShrinkArgs {
  const void *x;
  int64_t ldx;
  const void *A[LORA_MAX_SLICES];
  float *buf;
  MetaView mv;
  int list_off, list_cnt;   // segment list inside the work lists, and its count index
  int d_in, r_max, kc;      // kc: d_in rows per cluster CTA
  const int32_t *slot_rank;
  const float *slot_scale;
};

// NV = 16-byte vectors per A row (r_max / elements per vector).
template <typename TW, int NV>
__global__ void __launch_bounds__(kShrinkThreads) bgmv_shrink_kernel(ShrinkArgs a) {
  constexpr int VEC = Elem<TW>::kVec;
  constexpr int NRG = kShrinkThreads / NV;  // row groups
  extern __shared__ __align__(16) unsigned char smem[];
  const int cs = (int)cluster_nctarank(), crank = (int)cluster_ctarank();
  const int item = blockIdx.x / cs;
  const int slice = blockIdx.y;
  const int32_t *W = a.mv.work;
  if (item >= W[a.list_cnt]) return;  // the whole cluster leaves together
  const int seg = W[a.list_off + item];
  const int slot = a.mv.seg_slot[seg];
  const int cnt = a.mv.seg_count[seg];
  const int start = a.mv.seg_start[seg];
  const int r_max = a.r_max;
  const int r_a = min(max(a.slot_rank[slot], 0), r_max);
  const float scale = a.slot_scale[slot];
  const int j0 = crank * a.kc;
  const int len = max(0, min(a.d_in, j0 + a.kc) - j0);
  const TW *Ab = static_cast<const TW *>(a.A[slice]) + ((int64_t)slot * a.d_in + j0) * r_max;
  float *bufs = a.buf + (int64_t)slice * a.mv.num_tokens * r_max;

  TW *xs = reinterpret_cast<TW *>(smem);                                    // [kTT][kc]
  float *wpart = reinterpret_cast<float *>(smem + (size_t)kTT * a.kc * sizeof(TW));  // [warps][kTT][r_max]
  float *cpart = wpart + kShrinkWarps * kTT * r_max;                        // [kTT][r_max]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v = tid % NV, rg = tid / NV;
  const bool vactive = v * VEC < r_a;
  const int xv_row = len / VEC;

  for (int tok0 = 0; tok0 < cnt; tok0 += kTT) {
    const int nt = min(kTT, cnt - tok0);
    for (int i = tid; i < nt * xv_row; i += kShrinkThreads) {
      const int t = i / xv_row, c = i % xv_row;
      const int row = a.mv.sorted_rows[start + tok0 + t];
      const uint4 val = __ldg(reinterpret_cast<const uint4 *>(
          static_cast<const TW *>(a.x) + (int64_t)row * a.ldx + j0) + c);
      reinterpret_cast<uint4 *>(xs + t * a.kc)[c] = val;
    }
    __syncthreads();

    float acc[kTT][VEC];
#pragma unroll
    for (int t = 0; t < kTT; ++t)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[t][e] = 0.f;
    if (vactive) {
      constexpr int U = 4;
      for (int jb = rg; jb < len; jb += U * NRG) {
        uint4 av[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = jb + u * NRG;
          if (j < len) av[u] = __ldg(reinterpret_cast<const uint4 *>(Ab + (int64_t)j * r_max) + v);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = jb + u * NRG;
          if (j < len) {
            const TW *ap = reinterpret_cast<const TW *>(&av[u]);
            float af[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) af[e] = Elem<TW>::to_f(ap[e]);
#pragma unroll
            for (int t = 0; t < kTT; ++t) {
              if (t < nt) {
                const float xv = Elem<TW>::to_f(xs[t * a.kc + j]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[t][e] = fmaf(xv, af[e], acc[t][e]);
              }
            }
          }
        }
      }
    }
    // Reduce over the lanes that share this thread's vector column.
#pragma unroll
    for (int t = 0; t < kTT; ++t) {
      if (t < nt) {
#pragma unroll
        for (int o = NV; o < 32; o <<= 1)
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[t][e] += __shfl_xor_sync(0xffffffffu, acc[t][e], o);
      }
    }
    if (lane < NV) {
      for (int t = 0; t < nt; ++t)
#pragma unroll
        for (int e = 0; e < VEC; ++e) wpart[(warp * kTT + t) * r_max + v * VEC + e] = acc[t][e];
    }
    __syncthreads();
    for (int i = tid; i < nt * r_max; i += kShrinkThreads) {
      const int t = i / r_max, k = i % r_max;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kShrinkWarps; ++w) s += wpart[(w * kTT + t) * r_max + k];
      cpart[t * r_max + k] = s;
    }
    cluster_sync();
    if (crank == 0) {
      const int r4 = r_max / 4;
      for (int i = tid; i < nt * r4; i += kShrinkThreads) {
        const int t = i / r4, k = (i % r4) * 4;
        const uint32_t la = smem_addr(cpart + t * r_max + k);
        float4 s = ld_dsmem_f4(la, 0);
        for (int c = 1; c < cs; ++c) {
          const float4 p = ld_dsmem_f4(la, (uint32_t)c);
          s.x += p.x; s.y += p.y; s.z += p.z; s.w += p.w;
        }
        float4 o;
        o.x = (k + 0 < r_a) ? scale * s.x : 0.f;
        o.y = (k + 1 < r_a) ? scale * s.y : 0.f;
        o.z = (k + 2 < r_a) ? scale * s.z : 0.f;
        o.w = (k + 3 < r_a) ? scale * s.w : 0.f;
        const int row = a.mv.sorted_rows[start + tok0 + t];
        *reinterpret_cast<float4 *>(bufs + (int64_t)row * r_max + k) = o;
      }
    }
    cluster_sync();  // partials stay alive until CTA 0 has read them; buffers are reused next tile
  }
}

struct ExpandArgs {
  const float *buf;
  void *y;
  int64_t ldy;
  const void *B[LORA_MAX_SLICES];
  MetaView mv;
  int list_off, list_cnt;
  int r_max;
  int out_sizes[LORA_MAX_SLICES];
  int out_off[LORA_MAX_SLICES];
  int chunk_start[LORA_MAX_SLICES + 1];
  int n_slices;
  const int32_t *slot_rank;
};

template <typename TW, typename TY>
__global__ void __launch_bounds__(kExpandThreads) bgmv_expand_kernel(ExpandArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int32_t *W = a.mv.work;
  const int item = blockIdx.y;
  if (item >= W[a.list_cnt]) return;
  int s = 0;
  while (s + 1 < a.n_slices && (int)blockIdx.x >= a.chunk_start[s + 1]) ++s;
  const int out_s = a.out_sizes[s];
  const int n0 = ((int)blockIdx.x - a.chunk_start[s]) * kExpandCols + threadIdx.x * 8;
  const bool active = n0 < out_s;
  const int seg = W[a.list_off + item];
  const int slot = a.mv.seg_slot[seg];
  const int cnt = a.mv.seg_count[seg];
  const int start = a.mv.seg_start[seg];
  const int r_max = a.r_max;
  const int r_a = min(max(a.slot_rank[slot], 0), r_max);
  const TW *Bb = static_cast<const TW *>(a.B[s]) + (int64_t)slot * r_max * out_s + n0;
  const float *bufs = a.buf + (int64_t)s * a.mv.num_tokens * r_max;
  TY *y = static_cast<TY *>(a.y);

  float *us = reinterpret_cast<float *>(smem);   // [kTT][r_max]
  __shared__ int rows[kTT];

  for (int tok0 = 0; tok0 < cnt; tok0 += kTT) {
    const int nt = min(kTT, cnt - tok0);
    if (threadIdx.x < nt) rows[threadIdx.x] = a.mv.sorted_rows[start + tok0 + threadIdx.x];
    __syncthreads();
    for (int i = threadIdx.x; i < nt * r_max; i += kExpandThreads) {
      const int t = i / r_max, k = i % r_max;
      us[i] = (k < r_a) ? bufs[(int64_t)rows[t] * r_max + k] : 0.f;
    }
    __syncthreads();
    if (active) {
      float acc[kTT][8];
#pragma unroll
      for (int t = 0; t < kTT; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
      constexpr int U = 4;
      for (int kb = 0; kb < r_a; kb += U) {
        float bv[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (kb + u < r_a) load8_f32(Bb + (int64_t)(kb + u) * out_s, bv[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (kb + u < r_a) {
#pragma unroll
            for (int t = 0; t < kTT; ++t) {
              if (t < nt) {
                const float uk = us[t * r_max + kb + u];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[t][e] = fmaf(uk, bv[u][e], acc[t][e]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTT; ++t) {
        if (t < nt) {
          TY *yp = y + (int64_t)rows[t] * a.ldy + a.out_off[s] + n0;
          float yv[8];
          load8_rw(yp, yv);
#pragma unroll
          for (int e = 0; e < 8; ++e) yv[e] += acc[t][e];
          store8(yp, yv);
        }
      }
    }
    __syncthreads();
  }
}

int list_off_of(ListSel sel, int S) {
  return sel == kListSmall ? WorkLists::small_seg(S)
       : sel == kListLarge ? WorkLists::large_seg(S) : WorkLists::all_seg(S);
}
int list_cnt_of(ListSel sel) { return sel == kListSmall ? 1 : sel == kListLarge ? 2 : 0; }

template <typename TW, int NV>
cudaError_t shrink_nv(const ShrinkArgs &a, dim3 grid, size_t smem, int cs, cudaStream_t st) {
  auto k = bgmv_shrink_kernel<TW, NV>;
  cudaError_t e = set_max_dynamic_smem((const void *)k, 200 * 1024);
  if (e != cudaSuccess) return e;
  return launch_cluster(k, grid, dim3(kShrinkThreads), smem, st, (unsigned)cs, a);
}

}  // namespace

cudaError_t launch_bgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel,
                               const void *x, int64_t ldx, float *buf, cudaStream_t st) {
  const int max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  if (max_items <= 0) return cudaSuccess;
  ShrinkArgs a{};
  a.x = x;
  a.ldx = ldx;
  for (int s = 0; s < d.n_slices; ++s) a.A[s] = d.A[s];
  a.buf = buf;
  a.mv = mv;
  a.list_off = list_off_of(sel, mv.num_slots);
  a.list_cnt = list_cnt_of(sel);
  a.d_in = d.d_in;
  a.r_max = d.r_max;
  int cs = d.d_in / 512;
  cs = cs < 1 ? 1 : (cs > 8 ? 8 : cs);
  a.kc = ((d.d_in + cs - 1) / cs + 7) / 8 * 8;
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
  const size_t es = d.dtype == LORA_BF16 ? 2 : 4;
  const size_t smem = (size_t)kTT * a.kc * es + (size_t)(kShrinkWarps + 1) * kTT * d.r_max * sizeof(float);
  dim3 grid((unsigned)(cs * max_items), (unsigned)d.n_slices);
  if (d.dtype == LORA_BF16) {
    switch (d.r_max / 8) {
      case 1: return shrink_nv<__nv_bfloat16, 1>(a, grid, smem, cs, st);
      case 2: return shrink_nv<__nv_bfloat16, 2>(a, grid, smem, cs, st);
      case 4: return shrink_nv<__nv_bfloat16, 4>(a, grid, smem, cs, st);
      case 8: return shrink_nv<__nv_bfloat16, 8>(a, grid, smem, cs, st);
      case 16: return shrink_nv<__nv_bfloat16, 16>(a, grid, smem, cs, st);
    }
  } else {
    switch (d.r_max / 4) {
      case 2: return shrink_nv<float, 2>(a, grid, smem, cs, st);
      case 4: return shrink_nv<float, 4>(a, grid, smem, cs, st);
      case 8: return shrink_nv<float, 8>(a, grid, smem, cs, st);
      case 16: return shrink_nv<float, 16>(a, grid, smem, cs, st);
      case 32: return shrink_nv<float, 32>(a, grid, smem, cs, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel,
                               const float *buf, void *y, int64_t ldy, int y_dtype, cudaStream_t st) {
  const int max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  if (max_items <= 0) return cudaSuccess;
  ExpandArgs a{};
  a.buf = buf;
  a.y = y;
  a.ldy = ldy;
  a.mv = mv;
  a.list_off = list_off_of(sel, mv.num_slots);
  a.list_cnt = list_cnt_of(sel);
  a.r_max = d.r_max;
  a.n_slices = d.n_slices;
  int off = 0, chunks = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    a.B[s] = d.B[s];
    a.out_sizes[s] = d.out_sizes[s];
    a.out_off[s] = off;
    a.chunk_start[s] = chunks;
    off += d.out_sizes[s];
    chunks += (d.out_sizes[s] + kExpandCols - 1) / kExpandCols;
  }
  a.chunk_start[d.n_slices] = chunks;
  a.slot_rank = d.slot_rank;
  const size_t smem = (size_t)kTT * d.r_max * sizeof(float);
  dim3 grid((unsigned)chunks, (unsigned)max_items);
  if (d.dtype == LORA_BF16) {
    if (y_dtype == LORA_BF16)
      bgmv_expand_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kExpandThreads, smem, st>>>(a);
    else
      bgmv_expand_kernel<__nv_bfloat16, float><<<grid, kExpandThreads, smem, st>>>(a);
  } else {
    bgmv_expand_kernel<float, float><<<grid, kExpandThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ra
