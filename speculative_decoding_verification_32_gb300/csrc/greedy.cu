// greedy.cu -- greedy chain and tree verification (argmax match + margin rule).
//
// "Speculative Decoding: How a Small Model Speeds Up a Big One Without
// Changing Its Output", 'The Guarantee Behind Rejection Sampling': keep a
// draft iff it equals the target's argmax, else emit the argmax; 'Beyond Two
// Models: The EAGLE Line': a draft tree is verified in one pass and the best
// branch kept.  "Margins, Not Windows" section 3: a mismatched draft is
// promoted when p_target(draft) / p_target(top1) exceeds kappa.
//
// Only the target logits are read.  A persistent grid of warps streams
// (position, vocabulary slice) work items straight from HBM: each warp owns
// an item, keeps eight 16-byte loads per lane in flight, folds each vector to
// its largest element (packed bf16x2 max) and leaves the slice's largest
// logit and lowest index of it as a 16-byte partial -- no shared memory and
// no block barrier on the streaming path.  A second kernel, launched as a
// programmatic dependent, combines each row's partials (slices in vocabulary
// order, so ties keep the lowest index) with all its warps and walks the
// chain or the tree in one warp.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int kGWarps = kGreedyThreads / 32;
constexpr int kGU = 8;  // 16-byte vectors in flight per lane
constexpr int kWalkThreads = 256;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr float kInf = __builtin_huge_valf();

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
  // largest element of a vector; NaN if it holds one
  static __device__ __forceinline__ float vec_max(const uint32_t *w) {
    if constexpr (BF16) {
      const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(w[0], w[1]), bf16x2_max_nan(w[2], w[3]));
      return fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
      return fmax_nan(fmax_nan(__uint_as_float(w[0]), __uint_as_float(w[1])),
                      fmax_nan(__uint_as_float(w[2]), __uint_as_float(w[3])));
    }
  }
  // elements [v*EPV, v*EPV+EPV) of a slice starting at `src`; entries past
  // len are -inf.  VEC: one 16-byte load (the slice is whole vectors and
  // 16-byte aligned); otherwise element loads.
  template <bool VEC>
  static __device__ __forceinline__ void load_vec(uint32_t *w, const char *src, int v, int len,
                                                  uint64_t pol) {
    if constexpr (VEC) {
      const uint4 r = ld_stream_u4(src + (size_t)v * 16, pol);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
          const int e0 = v * 8 + 2 * i;
          const unsigned short *g = reinterpret_cast<const unsigned short *>(src);
          const uint32_t lo = e0 < len ? __ldg(g + e0) : 0xFF80u;
          const uint32_t hi = e0 + 1 < len ? __ldg(g + e0 + 1) : 0xFF80u;
          w[i] = lo | (hi << 16);
        } else {
          const int e = v * 4 + i;
          w[i] = e < len ? __ldg(reinterpret_cast<const unsigned int *>(src) + e) : 0xFF800000u;
        }
      }
    }
  }
};

// Combined (max, lowest argmax, flags) of one position from its slice
// partials, by one warp: each lane folds slices lane, lane+32, ... (in
// vocabulary order, so a later slice replaces only on a strictly larger
// value), then the warp takes the largest value and, among the lanes holding
// it, the lowest index.  A NaN partial is skipped; its flag marks the row.
__device__ __forceinline__ void combine_position(const GreedyPart *pp, int nslices, int lane,
                                                 float *mx, int *top, uint32_t *flags) {
  float best = -kInf;
  uint32_t bi = 0xFFFFFFFFu, f = 0;
  for (int s = lane; s < nslices; s += 32) {
    const int4 r = *reinterpret_cast<const int4 *>(pp + s);
    const float v = __int_as_float(r.x);
    f |= static_cast<uint32_t>(r.z);
    if (v > best) {
      best = v;
      bi = static_cast<uint32_t>(r.y);
    }
  }
  float M = best;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, o));
  bi = __reduce_min_sync(FULL_MASK, best == M ? bi : 0xFFFFFFFFu);
  f = __reduce_or_sync(FULL_MASK, f);
  if (M == kInf) f |= F_NONFINITE;
  else if (M == -kInf) f |= F_EMPTY;
  *mx = M;
  *top = bi == 0xFFFFFFFFu ? -1 : static_cast<int>(bi);
  *flags = f;
}

// Margin rule in fp64: l(draft) - l(top1) > T * ln(kappa).
__device__ __forceinline__ bool margin_promotes(float l_d, float l_top, float T, double ln_kappa) {
  return __dsub_rn((double)l_d, (double)l_top) > __dmul_rn((double)T, ln_kappa);
}

// Chain walk: draft j is kept iff it is position j's argmax (or promoted by
// the margin rule); the first miss emits that position's argmax, a full pass
// the bonus argmax.  mx_s / top_s / fl_s hold the combined positions, lg_s
// the draft token's logit at each position (loaded for the margin rule).
template <bool BF16>
__device__ void walk_greedy_chain(const GreedyParams &P, int b, int lane, const float *mx_s,
                                  const int *top_s, const uint32_t *fl_s, const float *lg_s) {
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
      const float mx = mx_s[j];
      const uint32_t f = fl_s[j];
      top = top_s[j];
      flags |= f;
      if (j < K && SV_INB((long long)b * K + j, (long long)P.B * K)) {
        const int y = __ldg(P.tokens + (size_t)b * K + j);
        if (y < 0 || y >= V) {
          flags |= F_BAD_TOKEN;
          ok = 0;
        } else if (y != top) {
          ok = P.use_margin && !f && margin_promotes(lg_s[j], mx, T, P.ln_kappa);
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
  for (int j = lane; j < npos && SV_INB(b, P.B); j += 32) {
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
// accepted node, lowest index on ties.  mx_s / top_s / fl_s hold the combined
// nodes, lg_s each node's token logit at its parent (for the margin rule);
// `scr` is shared scratch of 20 bytes per node.
template <bool BF16>
__device__ void walk_tree(const GreedyParams &P, int b, int lane, const float *mx_s, const int *top_s,
                          const uint32_t *fl_s, const float *lg_s, unsigned char *scr, int *shared_best) {
  const int N = P.npos, V = P.V;
  int *par_s = reinterpret_cast<int *>(scr);
  int *path_s = par_s + N;
  short *anc_s[2] = {reinterpret_cast<short *>(path_s + N), reinterpret_cast<short *>(path_s + N) + N};
  short *dep_s[2] = {anc_s[1] + N, anc_s[1] + 2 * N};
  unsigned char *ok_s = reinterpret_cast<unsigned char *>(dep_s[1] + N);
  unsigned char *acc_s[2] = {ok_s + N, ok_s + 2 * N};
  const int32_t *par_g = P.parent + (size_t)b * N;
  const int32_t *tok_g = P.tokens + (size_t)b * N;

  uint32_t flags = 0;
  float T = 1.0f;
  if (P.use_margin) {
    T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
    if (!(T > 0.f && T < kInf)) flags |= F_BAD_TEMPERATURE;
  }
  for (int i = lane; i < N; i += 32) {
    flags |= fl_s[i];
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
        ok = SV_INB(pa, N) &&
             (t == top_s[pa] || (P.use_margin && margin_promotes(lg_s[i], mx_s[pa], T, P.ln_kappa)));
      }
      ok_s[i] = static_cast<unsigned char>(ok);
    }
    __syncwarp();
    // Pointer jumping over the parent links: each round a node's link skips
    // twice as far toward the root, its flag becomes the AND of ok over the
    // path it spans and its depth the edges it spans (the root links to
    // itself with depth 0 and flag 1).  When every link is the root, a node
    // is accepted iff its whole root path is ok, and its depth is exact.
    int cur = 0;
    for (int i = lane; i < N; i += 32) {
      anc_s[0][i] = static_cast<short>(par_s[i]);
      dep_s[0][i] = static_cast<short>(i > 0 ? 1 : 0);
      acc_s[0][i] = i > 0 ? ok_s[i] : 1;
    }
    __syncwarp();
    for (int span = 1; span < N; span <<= 1) {
      bool more = false;
      for (int i = lane; i < N; i += 32) {
        const int p = SV_INB(anc_s[cur][i], N) ? anc_s[cur][i] : 0;
        const int pp = SV_INB(anc_s[cur][p], N) ? anc_s[cur][p] : 0;
        acc_s[cur ^ 1][i] = acc_s[cur][i] & acc_s[cur][p];
        dep_s[cur ^ 1][i] = static_cast<short>(dep_s[cur][i] + dep_s[cur][p]);
        anc_s[cur ^ 1][i] = static_cast<short>(pp);
        more |= pp != 0;
      }
      cur ^= 1;
      __syncwarp();
      if (!__any_sync(FULL_MASK, more)) break;
    }
    // the deepest accepted node, lowest index on ties (node 0 always counts)
    unsigned bk = 0;
    for (int i = lane; i < N; i += 32)
      if (acc_s[cur][i]) bk = max(bk, (static_cast<unsigned>(dep_s[cur][i]) << 16) | (0xFFFFu - i));
    bk = __reduce_max_sync(FULL_MASK, bk);
    if (lane == 0) {
      const int best = static_cast<int>(0xFFFFu - (bk & 0xFFFFu));
      const int d = static_cast<int>(bk >> 16);
      for (int n = best, k = d - 1; k >= 0 && SV_INB(n, N) && SV_INB(k, N); n = par_s[n], --k) path_s[k] = n;
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
        ot = SV_INB(pn, N) ? __ldg(tok_g + pn) : -1;
      } else if (i == d) {
        ot = SV_INB(best, N) ? top_s[best] : -1;
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

// Streaming pass: warp gw takes items gw, gw + GW, ... (item = position-major
// (position, slice)); per lane, U vectors are loaded before any is used.  A
// lane keeps the largest vector maximum it has seen (strictly larger
// replaces, so the earliest of its vectors wins a tie) with that vector's
// words; the warp then takes the largest value, the lowest vector index
// holding it, and that vector's first element equal to it.
template <bool BF16, bool VEC>
__global__ void __launch_bounds__(kGreedyThreads) greedy_kernel(const __grid_constant__ GreedyParams P) {
  using F = GFmt<BF16>;
  constexpr int EPV = F::EPV;
  constexpr int ESZ = F::ESZ;
  // let the walk kernel be scheduled now; it waits for this grid anyway
  allow_dependents();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kGWarps + (threadIdx.x >> 5);
  const int GW = gridDim.x * kGWarps;
  const int V = P.V, nsl = P.nslices;
  const int W = P.B * P.npos * nsl;
  const uint64_t pol = l2_policy_evict_first();
  for (int it = gw; it < W; it += GW) {
    const int pos = it / nsl;
    const int s0 = (it - pos * nsl) * P.slice;
    const int len = min(V - s0, P.slice);
    const int nvec = (len + EPV - 1) / EPV;
    const char *src = static_cast<const char *>(P.target) + ((size_t)pos * V + s0) * ESZ;
#ifdef SV_BOUNDS
    // the item's elements in the logits and its partial record; a bad item
    // is skipped (its row reads an old partial)
    if (!__all_sync(FULL_MASK, SV_INR((long long)pos * V + s0, len, (long long)P.B * P.npos * V) &&
                                   SV_INB(it, W)))
      continue;
#endif
    float best = -kInf, nan_acc = -kInf;
    int bv = -1;
    uint32_t wb[4] = {0u, 0u, 0u, 0u};
    for (int v0 = 0; v0 < nvec; v0 += 32 * kGU) {
      uint32_t w[kGU][4];
      if (v0 + 32 * kGU <= nvec) {  // every lane's vectors are in range
#pragma unroll
        for (int u = 0; u < kGU; ++u) F::template load_vec<VEC>(w[u], src, v0 + u * 32 + lane, len, pol);
      } else {
#pragma unroll
        for (int u = 0; u < kGU; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) {
            F::template load_vec<VEC>(w[u], src, v, len, pol);
          } else {
            w[u][0] = w[u][1] = w[u][2] = w[u][3] = BF16 ? 0xFF80FF80u : 0xFF800000u;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kGU; ++u) {
        const float vm = F::vec_max(w[u]);
        nan_acc = fmax_nan(nan_acc, vm);
        if (vm > best) {
          best = vm;
          bv = v0 + u * 32 + lane;
          wb[0] = w[u][0]; wb[1] = w[u][1]; wb[2] = w[u][2]; wb[3] = w[u][3];
        }
      }
    }
    float M = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, o));
    const uint32_t vmin =
        __reduce_min_sync(FULL_MASK, best == M ? static_cast<uint32_t>(bv) : 0xFFFFFFFFu);
    const bool nonfinite = __any_sync(FULL_MASK, nan_acc != nan_acc);
    // the lane holding the winning vector finds its first element equal to M
    const bool owner = vmin != 0xFFFFFFFFu && static_cast<uint32_t>(bv) == vmin && best == M;
    const unsigned who = __ballot_sync(FULL_MASK, owner);
    if (who == 0u) {  // every element is -inf
      if (lane == 0)
        P.part[it] = GreedyPart{nonfinite ? __int_as_float(0x7fc00000) : -kInf, -1,
                                nonfinite ? F_NONFINITE : 0u, 0};
    } else if (lane == __ffs(who) - 1) {
      int e = EPV - 1;
#pragma unroll
      for (int k = EPV - 1; k >= 0; --k)
        if (F::elem(wb, k) == M) e = k;
      P.part[it] = GreedyPart{nonfinite ? __int_as_float(0x7fc00000) : M,
                              s0 + static_cast<int>(vmin) * EPV + e, nonfinite ? F_NONFINITE : 0u, 0};
    }
  }
}

// One CTA per row: its warps combine the row's positions into shared memory,
// then warp 0 walks the chain or the tree.  Waits for the streaming kernel
// (programmatic dependent launch).
template <bool BF16>
__global__ void __launch_bounds__(kWalkThreads) greedy_walk_kernel(const __grid_constant__ GreedyParams P) {
  using F = GFmt<BF16>;
  extern __shared__ __align__(16) unsigned char wsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int npos = P.npos, V = P.V;
  int *best = reinterpret_cast<int *>(wsm);
  float *mx_s = reinterpret_cast<float *>(wsm + 16);
  int *top_s = reinterpret_cast<int *>(mx_s + npos);
  uint32_t *fl_s = reinterpret_cast<uint32_t *>(top_s + npos);
  float *lg_s = reinterpret_cast<float *>(fl_s + npos);
  // The margin rule's logits -- each draft token's (chain) or each node's
  // token at its parent (tree) -- are inputs the streaming kernel never
  // writes: load them before the dependency wait, so they arrive while the
  // stream finishes.  Out-of-range parents and tokens load nothing (the walk
  // flags the row).
  if (P.use_margin) {
    for (int i = threadIdx.x; i < npos; i += kWalkThreads) {
      float l = 0.f;
      if (P.tree) {
        const bool in = SV_INB((long long)b * npos + i, (long long)P.B * npos);
        const int pa = i > 0 && in ? __ldg(P.parent + (size_t)b * npos + i) : -1;
        const int t = i > 0 && in ? __ldg(P.tokens + (size_t)b * npos + i) : -1;
        if (pa >= 0 && pa < i && t >= 0 && t < V &&
            SV_INB(((long long)b * npos + pa) * V + t, (long long)P.B * npos * V))
          l = F::load_logit(P.target, ((size_t)b * npos + pa) * V + t);
      } else if (i < npos - 1 && SV_INB((long long)b * (npos - 1) + i, (long long)P.B * (npos - 1))) {
        const int y = __ldg(P.tokens + (size_t)b * (npos - 1) + i);
        if (y >= 0 && y < V && SV_INB(((long long)b * npos + i) * V + y, (long long)P.B * npos * V))
          l = F::load_logit(P.target, ((size_t)b * npos + i) * V + y);
      }
      lg_s[i] = l;
    }
  }
  grid_dependency_wait();
  // Each position's (max, lowest argmax, flags) from its slice partials, by
  // whichever mapping takes fewer dependent rounds of loads: a warp per
  // position (lanes over the slices; few positions with many slices, as in a
  // chain), or a thread per position with four partials in flight (many
  // positions, as in a tree).  Both take the largest value and, among the
  // slices holding it, the lowest index; NaN partials are skipped and flagged.
  const int nsl = P.nslices;
  const int by_warp = ((npos + kWalkWarps - 1) / kWalkWarps) * ((nsl + 31) / 32);
  const int by_thread = ((npos + kWalkThreads - 1) / kWalkThreads) * ((nsl + 3) / 4);
  if (by_warp <= by_thread) {
    for (int j = warp; j < npos; j += kWalkWarps) {
      float mx;
      int top;
      uint32_t f;
      if (!SV_INR(((long long)b * npos + j) * nsl, nsl, (long long)P.B * npos * nsl)) continue;
      combine_position(P.part + ((size_t)b * npos + j) * nsl, nsl, lane, &mx, &top, &f);
      if (lane == 0) {
        mx_s[j] = mx;
        top_s[j] = top;
        fl_s[j] = f;
      }
    }
  } else {
    // in vocabulary order, a later slice replacing only on a strictly larger
    // value
    for (int j = threadIdx.x; j < npos; j += kWalkThreads) {
      if (!SV_INR(((long long)b * npos + j) * nsl, nsl, (long long)P.B * npos * nsl)) continue;
      const GreedyPart *pp = P.part + ((size_t)b * npos + j) * nsl;
      float M = -kInf;
      uint32_t bi = 0xFFFFFFFFu, f = 0;
      auto fold = [&](const int4 &r) {
        const float v = __int_as_float(r.x);
        f |= static_cast<uint32_t>(r.z);
        if (v > M) {
          M = v;
          bi = static_cast<uint32_t>(r.y);
        }
      };
      int sl = 0;
      for (; sl + 4 <= nsl; sl += 4) {
        int4 r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = *reinterpret_cast<const int4 *>(pp + sl + q);
#pragma unroll
        for (int q = 0; q < 4; ++q) fold(r[q]);
      }
      for (; sl < nsl; ++sl) fold(*reinterpret_cast<const int4 *>(pp + sl));
      if (M == kInf) f |= F_NONFINITE;
      else if (M == -kInf) f |= F_EMPTY;
      mx_s[j] = M;
      top_s[j] = bi == 0xFFFFFFFFu ? -1 : static_cast<int>(bi);
      fl_s[j] = f;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  if (P.tree) walk_tree<BF16>(P, b, lane, mx_s, top_s, fl_s, lg_s, reinterpret_cast<unsigned char *>(lg_s + npos), best);
  else walk_greedy_chain<BF16>(P, b, lane, mx_s, top_s, fl_s, lg_s);
}

template <bool BF16, bool VEC>
void launch_stream(const GreedyParams &p, int grid, cudaStream_t s) {
  greedy_kernel<BF16, VEC><<<grid, kGreedyThreads, 0, s>>>(p);
}

}  // namespace

#ifdef SV_BOUNDS
SV_OOB_READER(oob_record_greedy)
#endif

cudaError_t launch_greedy(const GreedyParams &p, bool bf16, int grid, cudaStream_t s) {
  if (bf16) p.vec ? launch_stream<true, true>(p, grid, s) : launch_stream<true, false>(p, grid, s);
  else p.vec ? launch_stream<false, true>(p, grid, s) : launch_stream<false, false>(p, grid, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // walk: 16 bytes + 16 per position for the combined positions and the
  // margin logits, and 20 more per node for the tree walk's scratch
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B));
  cfg.blockDim = dim3(kWalkThreads);
  cfg.dynamicSmemBytes = 16 + static_cast<size_t>(p.npos) * (p.tree ? 36 : 16);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, greedy_walk_kernel<true>, p)
              : cudaLaunchKernelEx(&cfg, greedy_walk_kernel<false>, p);
}

cudaError_t greedy_max_blocks_per_sm(bool bf16, bool vec, int *blocks) {
  const void *k = bf16 ? (vec ? (const void *)greedy_kernel<true, true> : (const void *)greedy_kernel<true, false>)
                       : (vec ? (const void *)greedy_kernel<false, true> : (const void *)greedy_kernel<false, false>);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k, kGreedyThreads, 0);
}

}  // namespace sv
