// greedy.cu -- greedy chain and tree verification (argmax match + margin rule).
//
// "Speculative Decoding: How a Small Model Speeds Up a Big One Without
// Changing Its Output", 'The Guarantee Behind Rejection Sampling': keep a
// draft iff it equals the target's argmax, else emit the argmax; 'Beyond Two
// Models: The EAGLE Line': a draft tree is verified in one pass and the best
// branch kept.  "Margins, Not Windows" section 3: a mismatched draft is
// promoted when p_target(draft) / p_target(top1) exceeds kappa.
//
// Only the target logits are read.  A persistent grid streams (position,
// vocabulary slice) work items through a bulk-copy (TMA) ring in shared
// memory; each item leaves its slice's largest logit and lowest index of it
// as a 16-byte partial.  The CTA that completes the last item of a row
// combines the row's partials (slices in vocabulary order, so ties keep the
// lowest index) and walks the chain or the tree in one warp.
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int NT = kThreads;
constexpr int NW = NT / 32;
constexpr int kMaxStages = 8;
constexpr float kInf = __builtin_huge_valf();

struct alignas(16) GCtrl {
  uint64_t full[kMaxStages];
  uint64_t never;
  uint64_t pad0;
  float part_v[NW];
  int part_i[NW];
  uint32_t part_f[NW];
};
static_assert(sizeof(GCtrl) <= 1024, "control block must fit its reservation");

template <bool BF16>
struct GFmt {
  static constexpr int EPV = BF16 ? 8 : 4;
  static constexpr int ESZ = BF16 ? 2 : 4;
  static __device__ __forceinline__ float elem(const uint32_t *w, int e) {
    if constexpr (BF16) return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else return __uint_as_float(w[e]);
  }
  static __device__ __forceinline__ float load_logit(const void *base, size_t idx) {
    if constexpr (BF16)
      return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short *>(base) + idx)) << 16);
    else return __ldg(static_cast<const float *>(base) + idx);
  }
  // elements [v*EPV, v*EPV+EPV) of the slice; entries past len are -inf
  static __device__ __forceinline__ void load_vec(uint32_t *w, bool tma, const unsigned char *sbuf,
                                                  const char *gsrc, int v, int len) {
    if (tma) {
      uint4 r = ld_shared_u4(sbuf + (size_t)v * 16);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
          const int e0 = v * 8 + 2 * i;
          const unsigned short *g = reinterpret_cast<const unsigned short *>(gsrc);
          uint32_t lo = e0 < len ? __ldg(g + e0) : 0xFF80u;
          uint32_t hi = e0 + 1 < len ? __ldg(g + e0 + 1) : 0xFF80u;
          w[i] = lo | (hi << 16);
        } else {
          const int e = v * 4 + i;
          w[i] = e < len ? __ldg(reinterpret_cast<const unsigned int *>(gsrc) + e) : 0xFF800000u;
        }
      }
    }
  }
};

// (value, index) pair order: larger value first, then lower index.
__device__ __forceinline__ bool pair_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && (unsigned)i < (unsigned)bi);
}

// Combined (max, lowest argmax, flags) of one position from its slice partials.
__device__ __forceinline__ void combine_partials(const GreedyPart *pp, int nslices, float *mx,
                                                 int *top, uint32_t *flags) {
  float best = -kInf;
  int bi = -1;
  uint32_t f = 0;
  for (int s = 0; s < nslices; ++s) {
    const int4 r = *reinterpret_cast<const int4 *>(pp + s);
    const float v = __int_as_float(r.x);
    f |= static_cast<uint32_t>(r.z);
    if (v > best) {  // slices in vocabulary order: ties keep the earlier slice
      best = v;
      bi = r.y;
    }
  }
  if (best == kInf) f |= F_NONFINITE;
  else if (best == -kInf) f |= F_EMPTY;
  *mx = best;
  *top = bi;
  *flags = f;
}


// Margin rule in fp64: l(draft) - l(top1) > T * ln(kappa).
__device__ __forceinline__ bool margin_promotes(float l_d, float l_top, float T, double ln_kappa) {
  return __dsub_rn((double)l_d, (double)l_top) > __dmul_rn((double)T, ln_kappa);
}

template <bool BF16>
__device__ void walk_greedy_chain(const GreedyParams &P, int b, int lane) {
  using F = GFmt<BF16>;
  const int npos = P.npos, K = npos - 1, V = P.V;
  uint32_t flags = 0;
  float T = 1.0f;
  if (P.use_margin) {
    T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
    if (!(T > 0.f && T < kInf)) flags |= F_BAD_TEMPERATURE;
  }
  int stop = K, stop_top = -1, last_top = -1;
  for (int j0 = 0; j0 < npos; j0 += 32) {
    const int j = j0 + lane;
    int ok = 1, top = -1;
    if (j < npos) {
      float mx;
      uint32_t f;
      combine_partials(P.part + ((size_t)b * npos + j) * P.nslices, P.nslices, &mx, &top, &f);
      flags |= f;
      if (j < K) {
        const int y = __ldg(P.tokens + (size_t)b * K + j);
        if (y < 0 || y >= V) {
          flags |= F_BAD_TOKEN;
          ok = 0;
        } else if (y != top) {
          ok = P.use_margin && !f &&
               margin_promotes(F::load_logit(P.target, ((size_t)b * npos + j) * V + y), mx, T,
                               P.ln_kappa);
        }
      }
    }
    const unsigned fail = __ballot_sync(FULL_MASK, j < K && !ok);
    if (stop == K && fail) {
      const int src = __ffs(fail) - 1;
      stop = j0 + src;
      stop_top = __shfl_sync(FULL_MASK, top, src);
    }
    if (j0 + 32 >= npos) last_top = __shfl_sync(FULL_MASK, top, (npos - 1) - j0);
  }
  flags = __reduce_or_sync(FULL_MASK, flags);
  const int tok = stop == K ? last_top : stop_top;
  for (int j = lane; j < npos; j += 32) {
    int o = -1;
    if (!flags) o = j < stop ? __ldg(P.tokens + (size_t)b * K + j) : (j == stop ? tok : -1);
    P.out_tokens[(size_t)b * npos + j] = o;
  }
  if (lane == 0) {
    P.accepted_len[b] = flags ? -1 : stop;
    P.num_emitted[b] = flags ? 0 : stop + 1;
    P.row_status[b] = lowest_code(flags);
  }
}

// Tree walk: node i >= 1 is accepted iff its parent is accepted and its token
// is the parent's argmax (or promoted by the margin rule); keep the deepest
// accepted node, lowest index on ties.  `scr` is shared scratch for N nodes.
template <bool BF16>
__device__ void walk_tree(const GreedyParams &P, int b, int lane, unsigned char *scr, int *shared_best) {
  using F = GFmt<BF16>;
  const int N = P.npos, V = P.V;
  int *top_s = reinterpret_cast<int *>(scr);
  float *mx_s = reinterpret_cast<float *>(top_s + N);
  int *par_s = reinterpret_cast<int *>(mx_s + N);
  int *path_s = par_s + N;
  short *dep_s = reinterpret_cast<short *>(path_s + N);
  unsigned char *ok_s = reinterpret_cast<unsigned char *>(dep_s + N);
  unsigned char *acc_s = ok_s + N;
  const int32_t *par_g = P.parent + (size_t)b * N;
  const int32_t *tok_g = P.tokens + (size_t)b * N;

  uint32_t flags = 0;
  float T = 1.0f;
  if (P.use_margin) {
    T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
    if (!(T > 0.f && T < kInf)) flags |= F_BAD_TEMPERATURE;
  }
  for (int i = lane; i < N; i += 32) {
    float mx;
    int top;
    uint32_t f;
    combine_partials(P.part + ((size_t)b * N + i) * P.nslices, P.nslices, &mx, &top, &f);
    flags |= f;
    top_s[i] = top;
    mx_s[i] = mx;
    const int pa = __ldg(par_g + i);
    if (i == 0 ? pa != -1 : (pa < 0 || pa >= i)) flags |= F_BAD_PARENT;
    par_s[i] = (i == 0 || pa < 0 || pa >= i) ? 0 : pa;
    if (i > 0) {
      const int t = __ldg(tok_g + i);
      if (t < 0 || t >= V) flags |= F_BAD_TOKEN;
    }
  }
  flags = __reduce_or_sync(FULL_MASK, flags);
  __syncwarp();
  if (!flags) {
    for (int i = lane; i < N; i += 32) {
      int ok = 1;
      if (i > 0) {
        const int pa = par_s[i], t = __ldg(tok_g + i);
        ok = t == top_s[pa] ||
             (P.use_margin &&
              margin_promotes(F::load_logit(P.target, ((size_t)b * N + pa) * V + t), mx_s[pa], T,
                              P.ln_kappa));
      }
      ok_s[i] = static_cast<unsigned char>(ok);
    }
    __syncwarp();
    if (lane == 0) {
      acc_s[0] = 1;
      dep_s[0] = 0;
      int best = 0;
      for (int i = 1; i < N; ++i) {
        const int pa = par_s[i];
        acc_s[i] = acc_s[pa] & ok_s[i];
        dep_s[i] = static_cast<short>(dep_s[pa] + 1);
        if (acc_s[i] && dep_s[i] > dep_s[best]) best = i;
      }
      const int d = dep_s[best];
      for (int n = best, k = d - 1; k >= 0; n = par_s[n], --k) path_s[k] = n;
      shared_best[0] = best;
      shared_best[1] = d;
    }
    __syncwarp();
  }
  const int best = flags ? 0 : shared_best[0];
  const int d = flags ? -1 : shared_best[1];
  for (int i = lane; i < N; i += 32) {
    int pn = -1, ot = -1;
    if (!flags) {
      if (i < d) {
        pn = path_s[i];
        ot = __ldg(tok_g + pn);
      } else if (i == d) {
        ot = top_s[best];
      }
    }
    P.path_nodes[(size_t)b * N + i] = pn;
    P.out_tokens[(size_t)b * N + i] = ot;
  }
  if (lane == 0) {
    P.accepted_len[b] = flags ? -1 : d;
    P.num_emitted[b] = flags ? 0 : d + 1;
    P.row_status[b] = lowest_code(flags);
  }
  __syncwarp();
}

template <bool BF16>
__global__ void __launch_bounds__(NT, 1) greedy_kernel(const __grid_constant__ GreedyParams P) {
  using F = GFmt<BF16>;
  constexpr int EPV = F::EPV;
  constexpr int ESZ = F::ESZ;
  extern __shared__ __align__(128) unsigned char smem[];
  const int S = P.stages;
  GCtrl &ctl = *reinterpret_cast<GCtrl *>(smem + (size_t)S * P.buf_bytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int npos = P.npos, V = P.V, nsl = P.nslices;
  const int B = P.B;
  const int W = B * npos * nsl;
  const int G = (int)gridDim.x, g = (int)blockIdx.x;
  const int my_items = g < W ? (W - 1 - g) / G + 1 : 0;
  const bool tma = P.use_tma != 0;

  // let the walk kernel be scheduled now; it waits for this grid anyway
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&ctl.full[s], 1);
    mbar_init(&ctl.never, 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto geom = [&](int n, int &pos, int &s0, int &len) {
    const int it = g + n * G;
    pos = it / nsl;
    s0 = (it - pos * nsl) * P.slice;
    len = min(V - s0, P.slice);
  };
  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int n) {
    int pos, s0, len;
    geom(n, pos, s0, len);
    const int s = n % S;
    const uint32_t bytes = static_cast<uint32_t>(len) * ESZ;
    mbar_arrive_expect_tx(&ctl.full[s], bytes);
    bulk_g2s(smem + (size_t)s * P.buf_bytes,
             static_cast<const char *>(P.target) + ((size_t)pos * V + s0) * ESZ, bytes, &ctl.full[s],
             pol);
  };
  int issued = 0, n_break = -1;
  if (tma && tid == 0)
    for (; issued < min(S, my_items); ++issued) issue(issued);

  for (int n = 0; n < my_items; ++n) {
    int pos, s0, len;
    geom(n, pos, s0, len);
    const int s = n % S;
    const uint32_t parity = static_cast<uint32_t>(n / S) & 1u;
    bool timed_out = false;
    if (tma && n_break < 0)
      timed_out = P.force_timeout ? !mbar_wait_bounded(&ctl.never, 0u, P.wait_limit_ns)
                                  : !mbar_wait_bounded(&ctl.full[s], parity, P.wait_limit_ns);
    const unsigned char *sb = smem + (size_t)s * P.buf_bytes;
    const char *gsrc = static_cast<const char *>(P.target) + ((size_t)pos * V + s0) * ESZ;
    const int nvec = (len + EPV - 1) / EPV;
    float best = -kInf, nan_acc = -kInf;
    int bidx = -1;
    for (int v = tid; v < nvec; v += NT) {
      uint32_t w[4];
      F::load_vec(w, tma, sb, gsrc, v, len);
      const int valid = len - v * EPV;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = (e < valid) ? F::elem(w, e) : -kInf;
        nan_acc = fmax_nan(nan_acc, x);
        if (x > best) {
          best = x;
          bidx = v * EPV + e;
        }
      }
    }
    if (__syncthreads_or(timed_out) && n_break < 0) n_break = n;
    if (tma && tid == 0 && n_break < 0 && issued < my_items) issue(issued++);

    uint32_t f = (nan_acc != nan_acc) ? F_NONFINITE : 0u;
    if (n_break >= 0) f |= F_TIMEOUT;
    // block reduction of (best, lowest index), flags
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(FULL_MASK, best, o);
      const int oi = __shfl_xor_sync(FULL_MASK, bidx, o);
      if (pair_better(ov, oi, best, bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    f = __reduce_or_sync(FULL_MASK, f);
    if (lane == 0) {
      ctl.part_v[warp] = best;
      ctl.part_i[warp] = bidx;
      ctl.part_f[warp] = f;
    }
    __syncthreads();
    if (warp == 0) {
      best = lane < NW ? ctl.part_v[lane] : -kInf;
      bidx = lane < NW ? ctl.part_i[lane] : -1;
      f = lane < NW ? ctl.part_f[lane] : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, best, o);
        const int oi = __shfl_xor_sync(FULL_MASK, bidx, o);
        if (pair_better(ov, oi, best, bidx)) {
          best = ov;
          bidx = oi;
        }
      }
      f = __reduce_or_sync(FULL_MASK, f);
      if (lane == 0) {
        const int slice = (g + n * G) - pos * nsl;
        P.part[(size_t)pos * nsl + slice] =
            GreedyPart{best, bidx >= 0 ? s0 + bidx : -1, f, 0};
      }
    }
  }
  if (tma && n_break >= 0 && tid == 0)
    for (int m = n_break; m < issued; ++m)
      mbar_wait_bounded(&ctl.full[m % S], static_cast<uint32_t>(m / S) & 1u, P.wait_limit_ns);
}

// One warp per row: combine the row's partials and walk the chain or the
// tree.  Waits for the partial kernel (programmatic dependent launch).
template <bool BF16>
__global__ void greedy_walk_kernel(const __grid_constant__ GreedyParams P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(16) unsigned char wsm[];
  const int lane = threadIdx.x & 31;
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (b >= P.B) return;
  if (P.tree) {
    int *best = reinterpret_cast<int *>(wsm);
    walk_tree<BF16>(P, b, lane, wsm + 16, best);
  } else {
    walk_greedy_chain<BF16>(P, b, lane);
  }
}

// Set the shared-memory attribute once per device (again only if more is needed).
template <bool BF16>
cudaError_t prepare(size_t smem) {
  static std::atomic<size_t> done_smem[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done_smem[dev].load() >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(greedy_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e == cudaSuccess) done_smem[dev].store(smem);
  return e;
}

}  // namespace

cudaError_t launch_greedy(const GreedyParams &p, bool bf16, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = bf16 ? prepare<true>(smem) : prepare<false>(smem);
  if (e != cudaSuccess) return e;
  if (bf16) greedy_kernel<true><<<grid, NT, smem, s>>>(p);
  else greedy_kernel<false><<<grid, NT, smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // walk: trees need N*20 bytes of scratch per row, so one warp per block;
  // chains take four rows per block
  const int rows_per_block = p.tree ? 1 : 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.B + rows_per_block - 1) / rows_per_block));
  cfg.blockDim = dim3(static_cast<unsigned>(32 * rows_per_block));
  cfg.dynamicSmemBytes = p.tree ? 16 + static_cast<size_t>(p.npos) * 20 : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, greedy_walk_kernel<true>, p)
              : cudaLaunchKernelEx(&cfg, greedy_walk_kernel<false>, p);
}

cudaError_t greedy_max_blocks_per_sm(bool bf16, size_t smem, int *blocks) {
  cudaError_t e = bf16 ? prepare<true>(smem) : prepare<false>(smem);
  if (e != cudaSuccess) return e;
  return bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, greedy_kernel<true>, NT, smem)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, greedy_kernel<false>, NT, smem);
}

}  // namespace sv
