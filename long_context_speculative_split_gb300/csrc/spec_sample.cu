// Draft-token draw and modified rejection sampling over vocab-sized float32
// distributions.
//
// "Wann beschleunigt spekulatives Decoding das LLM-Serving?", section "Eine
// Verifizierungsrunde verstehen": candidates are accepted left to right using
// both distributions; at the first rejection a correction is drawn from the
// residual target distribution and later candidates are dropped; if all are
// accepted one more target token is drawn.  The paragraph after it: this
// preserves the target distribution.
//
// A draft step's draw of one draft row is one kernel (spec_draw_row: the
// statistics of every slice, then the CTA completing a sequence draws its
// token from the slice holding u * Z).  Otherwise two kernels per call:
//   1. spec_stats: (max, sum of exp) of every logit row the mode needs, each
//      row split over several small CTAs (HBM stream, float4 loads, full
//      occupancy);
//   2. spec_finish: one CTA of 1024 threads per sequence merges the row
//      statistics, tests all candidates at once (u1 * q(x) < p(x)) and keeps
//      the prefix before the first rejection, then draws the correction /
//      bonus (or, in draft mode, the draft token) by inverse CDF in two
//      levels: 32 warps each sum a contiguous slice of the weights, a
//      double-precision prefix over the 32 slice totals finds the slice
//      holding u * Z, and the whole block scans that slice to find the first
//      index whose running sum exceeds u * Z.  Softmax draws start from the
//      statistics slice that holds u * Z, so only that slice is read.
#include "common.cuh"

namespace mgd {
namespace {

constexpr int kStatThreads = 256;
constexpr int kThreads = 1024;  // finish kernel
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

struct StatParams {
  int B, gamma, V, split, nsplit, nrows;
  int r_begin, nr;  // rows [r_begin, r_begin + nr) of every sequence (unified row index)
};

// unified row r of sequence b: r <= gamma -> target row r, else draft row r - gamma - 1
__device__ __forceinline__ const float *row_ptr(const float *target, const float *draft, int b, int r, int gamma,
                                                int V) {
  if (r <= gamma) return target + (static_cast<size_t>(b) * (gamma + 1) + r) * V;
  return draft + (static_cast<size_t>(b) * gamma + (r - gamma - 1)) * V;
}

// (max, sum of exp(x - max)) of x[lo, hi) over a kStatThreads block; the
// result is valid in thread 0.  Rounds of 16 values per thread (all loads in
// flight), one update of the running max per round, then one FMA + exp2 + add
// per value.
template <bool VEC4>
__device__ float2 slice_stats(const float *__restrict__ x, int lo, int hi) {
  float m = -INFINITY, l = 0.f;
  auto round16 = [&](const float (&v)[16]) {
    float mx = v[0];
#pragma unroll
    for (int k = 1; k < 16; ++k) mx = fmaxf(mx, v[k]);
    if (mx > m) {
      l *= ex2((m - mx) * kLog2e);  // 0 while m is -inf
      m = mx;
    }
    if (m != -INFINITY) {
      const float ml = m * kLog2e;
#pragma unroll
      for (int k = 0; k < 16; ++k) l += ex2(fmaf(v[k], kLog2e, -ml));
    }
  };
  if (VEC4) {  // V % 4 == 0: a float4 is either wholly inside the slice or wholly past it
    for (int i = lo + 4 * threadIdx.x; i < hi; i += 16 * kStatThreads) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ii = i + u * 4 * kStatThreads;
        const float4 f = (ii < hi) ? __ldcs(reinterpret_cast<const float4 *>(x + ii))
                                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        v[4 * u] = f.x;
        v[4 * u + 1] = f.y;
        v[4 * u + 2] = f.z;
        v[4 * u + 3] = f.w;
      }
      round16(v);
    }
  } else {
    for (int i = lo + threadIdx.x; i < hi; i += 16 * kStatThreads) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int ii = i + u * kStatThreads;
        v[u] = (ii < hi) ? __ldcs(x + ii) : -INFINITY;
      }
      round16(v);
    }
  }
  // block reduce of (m, l)
  __shared__ float sm[2][kStatThreads / 32];
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    const float mu = (mn == -INFINITY) ? 0.f : mn;
    l = l * exp2f((m - mu) * kLog2e) + l2 * exp2f((m2 - mu) * kLog2e);
    m = mn;
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sm[0][w] = m;
    sm[1][w] = l;
  }
  __syncthreads();
  float2 r = make_float2(-INFINITY, 0.f);
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int i = 0; i < kStatThreads / 32; ++i) M = fmaxf(M, sm[0][i]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Lt = 0.f;
    for (int i = 0; i < kStatThreads / 32; ++i) Lt += sm[1][i] * exp2f((sm[0][i] - Mu) * kLog2e);
    r = make_float2(M, Lt);
  }
  return r;
}

template <bool VEC4>
__global__ void __launch_bounds__(kStatThreads) spec_stats_kernel(const float *__restrict__ target,
                                                                   const float *__restrict__ draft, StatParams sp,
                                                                   float2 *__restrict__ stats) {
  const int b = blockIdx.x / sp.nr;
  const int r = sp.r_begin + blockIdx.x % sp.nr;
  const int s = blockIdx.y;
  const int lo = s * sp.split;
  const float2 st = slice_stats<VEC4>(row_ptr(target, draft, b, r, sp.gamma, sp.V), lo, min(lo + sp.split, sp.V));
  if (threadIdx.x == 0) stats[(static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit + s] = st;
}

// One draft-token draw of a single draft row per sequence (a draft step):
// every CTA computes one slice's statistics; the CTA that completes a
// sequence's statistics (atomic ticket) draws its token.  The slice totals
// locate the slice holding u * Z; the block scans that slice: each thread sums
// a contiguous segment, warp scans order the threads, one warp turns the
// running double sum into a float target per warp, and the first thread whose
// range [excl, incl) holds the target walks its segment.
template <bool VEC4>
__global__ void __launch_bounds__(kStatThreads) spec_draw_row_kernel(const float *__restrict__ draft,
                                                                      int32_t *__restrict__ draft_tokens,
                                                                      const float *__restrict__ u, StatParams sp,
                                                                      float2 *__restrict__ stats,
                                                                      unsigned *__restrict__ tickets) {
  constexpr int kW = kStatThreads / 32;
  __shared__ int s_last, s_slice, s_tidx, s_lastpos;
  __shared__ float s_M, s_trel[kW], s_wsum[kW];
  __shared__ double s_pre;
  const int b = blockIdx.x, s = blockIdx.y;
  const int r = sp.r_begin;                // unified row index of the draft row
  const int row = r - sp.gamma - 1;        // its draft position
  const int V = sp.V;
  const float *x = draft + (static_cast<size_t>(b) * sp.gamma + row) * V;
  const float2 *st_b = stats + (static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit;
  {
    const int lo = s * sp.split;
    const float2 st = slice_stats<VEC4>(x, lo, min(lo + sp.split, V));
    if (threadIdx.x == 0) {
      stats[(static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit + s] = st;
      __threadfence();
      s_last = (atomicAdd(&tickets[b], 1u) == static_cast<unsigned>(sp.nsplit - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && sp.nsplit <= 32) {
    // the slice holding u * Z: every slice's (max, sum) loaded at once, one per
    // lane; float exponentials, double prefix sums across the lanes
    const float2 v = (lane < sp.nsplit) ? __ldcg(st_b + lane) : make_float2(-INFINITY, 0.f);
    float M = v.x;
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const double ts = (lane < sp.nsplit) ? static_cast<double>(v.y * exp2f((v.x - M) * kLog2e)) : 0.0;
    double incl = ts;
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double Z = __shfl_sync(0xffffffffu, incl, 31);
    const double tgt = static_cast<double>(u[(static_cast<size_t>(b) * (sp.gamma + 1) + row) * 3 + 0]) * Z;
    const unsigned hit = __ballot_sync(0xffffffffu, ts > 0.0 && incl > tgt);  // run + ts > tgt, run = incl - ts
    const unsigned mass = __ballot_sync(0xffffffffu, lane < sp.nsplit && v.y > 0.f);
    const int pick = hit ? (__ffs(hit) - 1) : (mass ? 31 - __clz(mass) : -1);
    const double run = __shfl_sync(0xffffffffu, incl - ts, pick < 0 ? 0 : pick);
    if (lane == 0) {
      s_M = M;
      s_slice = pick;
      s_pre = hit ? tgt - run : -1.0;  // rounding pushed u * Z past the total: the last slice with mass, its end
      s_tidx = 0x7fffffff;
      s_lastpos = -1;
    }
  } else if (threadIdx.x == 0 && sp.nsplit > 32) {  // the same, one slice at a time
    float M = -INFINITY;
    for (int q = 0; q < sp.nsplit; ++q) M = fmaxf(M, __ldcg(&st_b[q].x));
    double Z = 0.0;
    for (int q = 0; q < sp.nsplit; ++q) {
      const float2 v = __ldcg(st_b + q);
      Z += static_cast<double>(v.y * exp2f((v.x - M) * kLog2e));
    }
    const double tgt = static_cast<double>(u[(static_cast<size_t>(b) * (sp.gamma + 1) + row) * 3 + 0]) * Z;
    double run = 0.0;
    int pick = -1;
    for (int q = 0; q < sp.nsplit; ++q) {
      const float2 v = __ldcg(st_b + q);
      const double ts = static_cast<double>(v.y * exp2f((v.x - M) * kLog2e));
      if (ts > 0.0 && run + ts > tgt) {
        pick = q;
        break;
      }
      run += ts;
    }
    if (pick < 0) {  // rounding pushed u * Z past the total: the last slice with mass, its end
      for (int q = sp.nsplit - 1; q >= 0 && pick < 0; --q)
        if (__ldcg(&st_b[q].y) > 0.f) pick = q;
      run = tgt + 1.0;
    }
    s_M = M;
    s_slice = pick;
    s_pre = tgt - run;  // target measured from the slice start (negative: take its last entry)
    s_tidx = 0x7fffffff;
    s_lastpos = -1;
  }
  __syncthreads();
  const int pick_slice = s_slice;
  int tok = -1;
  if (pick_slice >= 0) {
    const float M = s_M;
    const int lo = pick_slice * sp.split, hi = min(lo + sp.split, V);
    const int seg = ((hi - lo + kStatThreads - 1) / kStatThreads + 3) / 4 * 4;  // contiguous entries per thread
    const int j0 = min(hi, lo + static_cast<int>(threadIdx.x) * seg), j1 = min(hi, j0 + seg);
    // 16 entries per batch, all loads in flight (segments start on a multiple of 4)
    auto load16 = [&](int jb, float (&v)[16]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int jj = jb + 4 * q;
        if (VEC4 && jj + 3 < j1) {
          const float4 f = __ldg(reinterpret_cast<const float4 *>(x + jj));
          v[4 * q] = f.x;
          v[4 * q + 1] = f.y;
          v[4 * q + 2] = f.z;
          v[4 * q + 3] = f.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 * q + e] = (jj + e < j1) ? __ldg(x + jj + e) : -INFINITY;
        }
      }
    };
    float tsum = 0.f;
    int lastpos = -1;
#pragma unroll 1
    for (int jb = j0; jb < j1; jb += 16) {
      float v[16];
      load16(jb, v);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float w = exp2f((v[k] - M) * kLog2e);
        tsum += w;
        if (w > 0.f) lastpos = jb + k;
      }
    }
    float incl = tsum;
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    if (lane == 31) s_wsum[warp] = incl;
    if (lastpos >= 0) atomicMax(&s_lastpos, lastpos);
    __syncthreads();
    if (warp == 0) {  // per-warp float targets from a double scan of the warp totals
      const double x0 = (lane < kW) ? static_cast<double>(s_wsum[lane]) : 0.0;
      double ix = x0;
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, ix, o);
        if (lane >= o) ix += y;
      }
      if (lane < kW) s_trel[lane] = fmaxf(0.f, static_cast<float>(s_pre - (ix - x0)));
    }
    __syncthreads();
    const float trel = s_trel[warp];
    if (tsum > 0.f && excl <= trel && incl > trel && s_pre >= 0.0) atomicMin(&s_tidx, static_cast<int>(threadIdx.x));
    __syncthreads();
    if (static_cast<int>(threadIdx.x) == s_tidx) {
      float c = excl;
      int p = -1;
#pragma unroll 1
      for (int jb = j0; jb < j1 && p < 0; jb += 16) {
        float v[16];
        load16(jb, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float w = exp2f((v[k] - M) * kLog2e);
          c += w;
          if (p < 0 && w > 0.f && c > trel) p = jb + k;
        }
      }
      s_lastpos = (p >= 0) ? p : lastpos;  // the crossing is here; rounding: this segment's last positive weight
    }
    __syncthreads();
    tok = s_lastpos;  // no claim: the target lies past the slice's scanned total (rounding): its last entry
  }
  if (threadIdx.x == 0) {
    draft_tokens[static_cast<size_t>(b) * sp.gamma + row] = tok;
    tickets[b] = 0u;  // left clean for the next call on this workspace (the call also clears it first)
  }
}

// Weights of a draw: MODE 0 -> exp(a - Ma) (an unnormalised softmax);
// MODE 1 -> max(0, exp(a - Ma) * ia - exp(c - Mc) * ic) (residual p - q).
struct DrawSrc {
  const float *a;
  const float *c;
  float Ma, ia, Mc, ic;
  int mode;
};

__device__ __forceinline__ float weight_of(const DrawSrc &s, float a, float c) {
  const float pa = exp2f((a - s.Ma) * kLog2e);
  if (s.mode == 0) return pa;
  const float pc = exp2f((c - s.Mc) * kLog2e);
  return fmaxf(0.f, pa * s.ia - pc * s.ic);
}

// Weights of entries i..i+3 (zero at or past `hi`).  With VEC4, i is a
// multiple of 4 and the rows are 16-byte aligned.
template <bool VEC4>
__device__ __forceinline__ void weights4(const DrawSrc &s, int i, int hi, float (&w)[4]) {
  float a[4], c[4] = {0.f, 0.f, 0.f, 0.f};
  if (VEC4 && i + 3 < hi) {
    const float4 fa = __ldg(reinterpret_cast<const float4 *>(s.a + i));
    a[0] = fa.x;
    a[1] = fa.y;
    a[2] = fa.z;
    a[3] = fa.w;
    if (s.mode == 1) {
      const float4 fc = __ldg(reinterpret_cast<const float4 *>(s.c + i));
      c[0] = fc.x;
      c[1] = fc.y;
      c[2] = fc.z;
      c[3] = fc.w;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = weight_of(s, a[e], c[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i + e < hi) {
        a[e] = __ldg(s.a + i + e);
        if (s.mode == 1) c[e] = __ldg(s.c + i + e);
        w[e] = weight_of(s, a[e], c[e]);
      } else {
        w[e] = 0.f;
      }
    }
  }
}

struct DrawShared {
  float tot[kWarps];
  int last[kWarps];
  float wsum[kWarps];
  float trel[kWarps];
  double base;
  double target;
  double chunk;
  int wstar;
  int tidx;  // first thread of the block-wide scan holding the crossing
  int idx;
  int status;  // 0 ok, 1 total weight is zero
};

// Block-wide inverse-CDF draw over the index range [r0, r1).  The target is
// u * (sum of the weights in the range) when `target_in` < 0, else
// `target_in` (a running-sum value measured from r0).  Returns the index, or
// -1 when the weights of the range sum to zero.
template <bool VEC4>
__device__ int block_draw(const DrawSrc &src, int r0, int r1, float u, double target_in, DrawShared &sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = r1 - r0;
  const int per = ((n + kWarps * 128 - 1) / (kWarps * 128)) * 128;  // slice per warp, multiple of 128
  {
    const int lo = r0 + warp * per, hi = min(lo + per, r1);
    float sum = 0.f;
    int last = -1;
#pragma unroll 4
    for (int i = lo + 4 * lane; i < hi; i += 128) {
      float w[4];
      weights4<VEC4>(src, i, hi, w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sum += w[e];
        if (w[e] > 0.f) last = i + e;
      }
    }
    sum = warp_sum_xor(sum, 1, 16);
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0) {
      sh.tot[warp] = sum;
      sh.last[warp] = last;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double Z = 0.0;
    for (int w = 0; w < kWarps; ++w) Z += static_cast<double>(sh.tot[w]);
    sh.status = (Z > 0.0) ? 0 : 1;
    const double target = (target_in < 0.0) ? static_cast<double>(u) * Z : target_in;
    double run = 0.0;
    int ws = -1;
    double base = 0.0;
    for (int w = 0; w < kWarps; ++w) {
      if (sh.tot[w] > 0.f && run + static_cast<double>(sh.tot[w]) > target) {
        ws = w;
        base = run;
        break;
      }
      run += static_cast<double>(sh.tot[w]);
    }
    if (ws < 0) {  // rounding pushed u*Z past the total: last slice with mass, its last entry
      for (int w = kWarps - 1; w >= 0; --w)
        if (sh.tot[w] > 0.f) {
          ws = w;
          break;
        }
      base = target + 1.0;
    }
    sh.wstar = ws;
    sh.base = base;
    sh.target = target;
    sh.idx = 0x7fffffff;
  }
  __syncthreads();
  if (sh.status != 0) return -1;
  // Second level: the whole block scans slice wstar, 4 * kThreads entries at a
  // time.  Double precision is rare on this GPU, so one warp turns the running
  // sum into a float target relative to each warp's start (clamped at 0);
  // within a warp, thread t covers [excl_t, incl_t) and neighbours share their
  // endpoints exactly, so a target inside the chunk is claimed by at least one
  // thread, and the first claiming thread holds the crossing.
  const int ws = sh.wstar;
  const int lo = r0 + ws * per, hi = min(lo + per, r1);
  if (sh.base <= sh.target) {
    for (int c0 = lo; c0 < hi; c0 += 4 * kThreads) {
      const int i = c0 + 4 * threadIdx.x;
      float w[4];
      weights4<VEC4>(src, i, hi, w);
      const float ls = (w[0] + w[1]) + (w[2] + w[3]);
      float incl = ls;
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.f;
      if (lane == 31) sh.wsum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const double x = static_cast<double>(sh.wsum[lane]);
        double ix = x;  // inclusive prefix of the warp totals
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, ix, o);
          if (lane >= o) ix += y;
        }
        double ex = __shfl_up_sync(0xffffffffu, ix, 1);
        if (lane == 0) ex = 0.0;
        sh.trel[lane] = fmaxf(0.f, static_cast<float>(sh.target - (sh.base + ex)));
        if (lane == 31) sh.chunk = ix;
        if (lane == 0) sh.tidx = 0x7fffffff;
      }
      __syncthreads();
      const float trel = sh.trel[warp];
      if (ls > 0.f && excl <= trel && incl > trel) atomicMin(&sh.tidx, static_cast<int>(threadIdx.x));
      __syncthreads();
      const int tsel = sh.tidx;
      if (static_cast<int>(threadIdx.x) == tsel) {
        float cacc = excl;
        int pick = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          cacc += w[e];
          if (pick < 0 && w[e] > 0.f && cacc > trel) pick = i + e;
        }
        if (pick < 0)  // the crossing is here but rounding moved it: last positive weight
          for (int e = 3; e >= 0; --e)
            if (w[e] > 0.f) {
              pick = i + e;
              break;
            }
        sh.idx = pick;
      }
      if (threadIdx.x == 0 && tsel == 0x7fffffff) sh.base += sh.chunk;  // next chunk
      __syncthreads();
      if (tsel != 0x7fffffff) break;
    }
  }
  if (threadIdx.x == 0 && sh.idx == 0x7fffffff) sh.idx = sh.last[ws];
  __syncthreads();
  return sh.idx;
}

// Draw from softmax(row) knowing the per-slice statistics of the row (slices of
// `split` entries): the slice totals locate the slice holding u * Z, and only
// that slice is scanned.
template <bool VEC4>
__device__ int draw_softmax_row(const float *row, const float2 *st, int nsplit, int split, int V, float M, float u,
                                DrawShared &sh, double *s_pre, int *s_slice) {
  if (threadIdx.x == 0) {
    double Z = 0.0;
    for (int s = 0; s < nsplit; ++s) Z += static_cast<double>(st[s].y * exp2f((st[s].x - M) * kLog2e));
    const double target = static_cast<double>(u) * Z;
    double run = 0.0;
    int pick = nsplit - 1;
    for (int s = 0; s < nsplit; ++s) {
      const double ts = static_cast<double>(st[s].y * exp2f((st[s].x - M) * kLog2e));
      if (ts > 0.0 && run + ts > target) {
        pick = s;
        break;
      }
      run += ts;
    }
    if (run > target) run = target;  // only when every later slice is empty
    *s_pre = target - run;
    *s_slice = pick;
  }
  __syncthreads();
  const int s = *s_slice;
  const double t = *s_pre;
  DrawSrc src{row, nullptr, M, 1.f, 0.f, 0.f, 0};
  const int r0 = s * split, r1 = min(V, r0 + split);
  int tok = block_draw<VEC4>(src, r0, r1, u, t, sh);
  if (tok < 0) tok = block_draw<VEC4>(src, 0, V, u, -1.0, sh);  // the slice held no mass: full scan
  return tok;
}

__device__ __forceinline__ void merge_stats(const float2 *st, int nsplit, float &M, float &Z) {
  M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, st[s].x);
  Z = 0.f;
  for (int s = 0; s < nsplit; ++s) Z += st[s].y * exp2f((st[s].x - M) * kLog2e);
}

template <bool VEC4>
__global__ void __launch_bounds__(kThreads, 1) spec_finish_kernel(const float *__restrict__ target,
                                                               const float *__restrict__ draft,
                                                               int32_t *__restrict__ draft_tokens,
                                                               const float *__restrict__ u, StatParams sp, int mode,
                                                               int32_t *__restrict__ out_tokens,
                                                               int32_t *__restrict__ num_accepted,
                                                               const float2 *__restrict__ stats, WsHeader *hdr) {
  __shared__ float sM[33], sZ[33];
  __shared__ int s_last, s_slice;
  __shared__ int s_tok[16];
  __shared__ unsigned char s_ok[16], s_bad[16];
  __shared__ double s_pre;
  __shared__ DrawShared sh;
  const int b = blockIdx.x;
  const int g = sp.gamma, V = sp.V;

  for (int r = sp.r_begin + threadIdx.x; r < sp.r_begin + sp.nr; r += kThreads)
    merge_stats(stats + (static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit, sp.nsplit, sM[r], sZ[r]);
  __syncthreads();

  if (mode == 1) {  // draft draw: row s uses draft row s, uniform slot 0
    for (int r = sp.r_begin; r < sp.r_begin + sp.nr; ++r) {
      const int s = r - g - 1;
      const float uu = u[(static_cast<size_t>(b) * (g + 1) + s) * 3 + 0];
      const int tok = draw_softmax_row<VEC4>(row_ptr(target, draft, b, r, g, V),
                                             stats + (static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit, sp.nsplit,
                                             sp.split, V, sM[r], uu, sh, &s_pre, &s_slice);
      if (threadIdx.x == 0) draft_tokens[static_cast<size_t>(b) * g + s] = tok;
      __syncthreads();
    }
    return;
  }

  // every candidate's test at once; the chain keeps the prefix before the first rejection
  if (threadIdx.x < g) {
    const int i = threadIdx.x;
    const int x = draft_tokens[static_cast<size_t>(b) * g + i];
    const bool bad = (x < 0 || x >= V);
    bool acc = false;
    if (!bad) {
      const float *t = row_ptr(target, draft, b, i, g, V);
      const float *d = row_ptr(target, draft, b, g + 1 + i, g, V);
      const float px = exp2f((t[x] - sM[i]) * kLog2e) / sZ[i];
      const float qx = exp2f((d[x] - sM[g + 1 + i]) * kLog2e) / sZ[g + 1 + i];
      const float u1 = u[(static_cast<size_t>(b) * (g + 1) + i) * 3 + 1];
      acc = (u1 * qx < px);
    }
    s_tok[i] = x;
    s_ok[i] = acc ? 1 : 0;
    s_bad[i] = bad ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = g;
    for (int i = 0; i < g; ++i) {
      if (s_bad[i]) {
        raise_error(hdr, 0x4u);
        j = i;
        break;
      }
      if (!s_ok[i]) {
        j = i;
        break;
      }
      out_tokens[static_cast<size_t>(b) * (g + 1) + i] = s_tok[i];
    }
    s_last = j;
    num_accepted[b] = j;
  }
  __syncthreads();
  const int j = s_last;
  const float uu = u[(static_cast<size_t>(b) * (g + 1) + j) * 3 + 2];
  int tok;
  if (j < g) {
    DrawSrc src{row_ptr(target, draft, b, j, g, V), row_ptr(target, draft, b, g + 1 + j, g, V), sM[j],
                1.f / sZ[j], sM[g + 1 + j], 1.f / sZ[g + 1 + j], 1};
    tok = block_draw<VEC4>(src, 0, V, uu, -1.0, sh);
    if (tok < 0) {  // the residual vanished through rounding: draw from p_j
      DrawSrc sp2{row_ptr(target, draft, b, j, g, V), nullptr, sM[j], 1.f, 0.f, 0.f, 0};
      tok = block_draw<VEC4>(sp2, 0, V, uu, -1.0, sh);
    }
  } else {  // bonus from p_gamma
    tok = draw_softmax_row<VEC4>(row_ptr(target, draft, b, g, g, V),
                                 stats + (static_cast<size_t>(b) * sp.nrows + g) * sp.nsplit, sp.nsplit, sp.split, V,
                                 sM[g], uu, sh, &s_pre, &s_slice);
  }
  if (threadIdx.x == 0) {
    out_tokens[static_cast<size_t>(b) * (g + 1) + j] = tok;
    for (int i = j + 1; i <= g; ++i) out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
  }
}

}  // namespace

SpecPlan plan_spec(int B, int gamma, int V) {
  SpecPlan p{};
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.split = 16384;
  p.nsplit = (V + p.split - 1) / p.split;
  p.nrows = 2 * gamma + 1;
  p.off_tickets = kAlign;
  p.off_stats = align_up(p.off_tickets + sizeof(unsigned) * static_cast<size_t>(B));
  p.ws_bytes = align_up(p.off_stats + sizeof(float2) * static_cast<size_t>(B) * p.nrows * p.nsplit);
  return p;
}

cudaError_t launch_spec(const SpecPlan &p, const SpecArgs &a) {
  cudaError_t e = cudaMemsetAsync(a.ws, 0, p.off_stats, a.stream);  // header and tickets
  if (e != cudaSuccess) return e;
  StatParams sp;
  sp.B = p.B;
  sp.gamma = p.gamma;
  sp.V = p.V;
  sp.split = p.split;
  sp.nsplit = p.nsplit;
  sp.nrows = p.nrows;
  if (a.mode == 0) {
    sp.r_begin = 0;
    sp.nr = p.nrows;
  } else if (a.row < 0) {
    sp.r_begin = p.gamma + 1;
    sp.nr = p.gamma;
  } else {
    sp.r_begin = p.gamma + 1 + a.row;
    sp.nr = 1;
  }
  float2 *stats = reinterpret_cast<float2 *>(static_cast<unsigned char *>(a.ws) + p.off_stats);
  WsHeader *hdr = static_cast<WsHeader *>(a.ws);
  const bool vec4 = (p.V % 4) == 0 && (reinterpret_cast<uintptr_t>(a.draft) % 16) == 0 &&
                    (a.target == nullptr || (reinterpret_cast<uintptr_t>(a.target) % 16) == 0);
  if (a.mode == 1 && a.row >= 0) {  // one draft row: statistics and draw in one launch
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(a.ws) + p.off_tickets);
    const dim3 g(p.B, p.nsplit);
    if (vec4)
      spec_draw_row_kernel<true><<<g, kStatThreads, 0, a.stream>>>(a.draft, a.draft_tokens, a.u, sp, stats, tickets);
    else
      spec_draw_row_kernel<false><<<g, kStatThreads, 0, a.stream>>>(a.draft, a.draft_tokens, a.u, sp, stats,
                                                                     tickets);
    return cudaGetLastError();
  }
  dim3 g1(p.B * sp.nr, p.nsplit);
  if (vec4)
    spec_stats_kernel<true><<<g1, kStatThreads, 0, a.stream>>>(a.target, a.draft, sp, stats);
  else
    spec_stats_kernel<false><<<g1, kStatThreads, 0, a.stream>>>(a.target, a.draft, sp, stats);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (vec4)
    spec_finish_kernel<true><<<p.B, kThreads, 0, a.stream>>>(a.target, a.draft, a.draft_tokens, a.u, sp, a.mode,
                                                             a.out_tokens, a.num_accepted, stats, hdr);
  else
    spec_finish_kernel<false><<<p.B, kThreads, 0, a.stream>>>(a.target, a.draft, a.draft_tokens, a.u, sp, a.mode,
                                                              a.out_tokens, a.num_accepted, stats, hdr);
  return cudaGetLastError();
}

}  // namespace mgd
