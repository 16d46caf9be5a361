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
// Every draw is an inverse-CDF draw in three levels over a vocab row: the row
// is cut into sub-ranges of 2048 entries (one warp each), whose weight sums
// locate the sub-range holding u * Z; the CTA that completes a sequence scans
// only that sub-range, 8 entries per thread held in registers, with a block
// scan ordering the threads.  Sums of sub-range weights are float; their
// running prefix is double.
//
//   spec_draw_row: a draft step's draw of one draft row per sequence.  Every
//     warp streams one sub-range and records its (max, sum of exp); the CTA
//     completing a sequence (atomic ticket) merges the sub-range records and
//     draws.  Each CTA also leaves its chunk's (max, sum of exp) of the row
//     in the workspace, and the drawing CTA marks the row as drawn, so that
//     the round's rejection sample need not stream the draft rows again.
//     One launch.
//   spec_stats + spec_decide: rejection sampling.  spec_stats computes
//     (max, sum of exp) of each 16384-entry slice of every target row, and of
//     every draft row unless the draws of the round left theirs
//     (MGD_VERIFY_DRAWN: the decision kernel checks the marks and clears them);
//     spec_decide runs over (sequence, 16384-entry chunk): every CTA of a
//     sequence merges the row statistics and takes the same acceptance
//     decisions (u * q(x) < p(x) for each candidate, the chain keeps the prefix
//     before the first rejection), then sums the weights of the final draw --
//     the residual max(0, p - q) at the first rejection (and p itself, in case
//     the residual vanishes through rounding), or p of the bonus row -- over its
//     chunk, one warp per sub-range; the CTA completing the sequence draws.
//
// No clearing launch: the tickets go back to zero when a sequence completes,
// and the workspace header resets itself at the last completing CTA's check-in.
#include "common.cuh"

namespace mgd {
namespace {

constexpr int kStatThreads = 256;
constexpr int kWarps = kStatThreads / 32;
constexpr int kSub = 2048;                 // entries per sub-range (one warp)
constexpr int kChunk = kWarps * kSub;      // entries per CTA of the draw kernels (= the statistics split)
constexpr int kRecSmem = 512;              // sub-range records a completing CTA stages in shared memory
constexpr float kLog2e = 1.4426950408889634f;

struct StatParams {
  int B, gamma, V, split, nsplit, nrows, nsub;
  int r_begin, nr;  // rows [r_begin, r_begin + nr) of every sequence (unified row index)
  int reuse;        // rejection sample: the draft rows' statistics come from this round's draws
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
  __shared__ float sm[2][kWarps];
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
    for (int i = 0; i < kWarps; ++i) M = fmaxf(M, sm[0][i]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Lt = 0.f;
    for (int i = 0; i < kWarps; ++i) Lt += sm[1][i] * exp2f((sm[0][i] - Mu) * kLog2e);
    r = make_float2(M, Lt);
  }
  return r;
}

template <bool VEC4>
__global__ void __launch_bounds__(kStatThreads) spec_stats_kernel(const float *__restrict__ target,
                                                                   const float *__restrict__ draft, StatParams sp,
                                                                   float2 *__restrict__ stats) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x / sp.nr;
  const int r = sp.r_begin + blockIdx.x % sp.nr;
  const int s = blockIdx.y;
  const int lo = s * sp.split;
  const float2 st = slice_stats<VEC4>(row_ptr(target, draft, b, r, sp.gamma, sp.V), lo, min(lo + sp.split, sp.V));
  if (threadIdx.x == 0) stats[(static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit + s] = st;
}

// Weights of a draw, as a function of the entry index: kind 0 -> exp(a - Ma) *
// ia (a softmax); kind 1 -> max(0, exp(a - Ma) * ia - exp(c - Mc) * ic) (the
// residual p - q).  ia, ic are the reciprocal normalisers.
struct Weights {
  const float *a;
  const float *c;
  float Ma, ia, Mc, ic;
  int kind;
  __device__ __forceinline__ float operator()(float av, float cv) const {
    const float pa = exp2f((av - Ma) * kLog2e) * ia;
    if (kind == 0) return pa;
    return fmaxf(0.f, pa - exp2f((cv - Mc) * kLog2e) * ic);
  }
};

// The 8 entries [i, i + 8) of a weight row (zero at or past `hi`).  With VEC4,
// i is a multiple of 8 and the rows are 16-byte aligned.
template <bool VEC4>
__device__ __forceinline__ void weights8(const Weights &w, int i, int hi, float (&out)[8]) {
  float a[8], c[8];
  if (VEC4 && i + 7 < hi) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 fa = __ldg(reinterpret_cast<const float4 *>(w.a + i + 4 * h));
      a[4 * h] = fa.x, a[4 * h + 1] = fa.y, a[4 * h + 2] = fa.z, a[4 * h + 3] = fa.w;
      if (w.kind == 1) {
        const float4 fc = __ldg(reinterpret_cast<const float4 *>(w.c + i + 4 * h));
        c[4 * h] = fc.x, c[4 * h + 1] = fc.y, c[4 * h + 2] = fc.z, c[4 * h + 3] = fc.w;
      } else {
        c[4 * h] = c[4 * h + 1] = c[4 * h + 2] = c[4 * h + 3] = 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = w(a[e], c[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (i + e < hi) {
        a[e] = __ldg(w.a + i + e);
        c[e] = (w.kind == 1) ? __ldg(w.c + i + e) : 0.f;
        out[e] = w(a[e], c[e]);
      } else {
        out[e] = 0.f;
      }
    }
  }
}

struct DrawShared {
  double pre;      // weight before the chosen sub-range, subtracted from the target
  int sub;         // chosen sub-range, -1 if every weight is zero
  int tidx;        // first thread whose range holds the target
  int tok;
  float wsum[kWarps];
  float trel[kWarps];
};

// Warp 0: pick the sub-range holding u * Z among n sub-ranges of weight
// wsum(q) (a function evaluated the same way on every call).  Lane L sums a
// contiguous block of sub-ranges, a double scan over the lanes locates the
// block holding the target, and that lane walks its block.  Sets sh.sub (-1
// when Z == 0) and sh.pre (the target measured from the sub-range start); a
// target past the total (rounding) picks the last sub-range with weight with
// sh.pre = -1, so that its last entry with weight is drawn.
template <typename F>
__device__ __forceinline__ void pick_sub(F wsum, int n, float u, DrawShared &sh) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  const int q0 = min(n, lane * per), q1 = min(n, q0 + per);
  double ls = 0.0;
  for (int q = q0; q < q1; ++q) ls += static_cast<double>(wsum(q));
  double incl = ls;
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const double Z = __shfl_sync(0xffffffffu, incl, 31);
  const double tgt = static_cast<double>(u) * Z;
  const unsigned hit = __ballot_sync(0xffffffffu, ls > 0.0 && incl > tgt);
  const unsigned mass = __ballot_sync(0xffffffffu, ls > 0.0);
  if (lane == 0) sh.sub = -1;
  __syncwarp();
  if (hit) {
    if (lane == __ffs(hit) - 1) {
      double run = incl - ls;
      int pick = -1, last = -1;
      for (int q = q0; q < q1 && pick < 0; ++q) {
        const double w = static_cast<double>(wsum(q));
        if (w > 0.0) {
          last = q;
          if (run + w > tgt) pick = q;
          else run += w;
        }
      }
      sh.sub = pick >= 0 ? pick : last;
      sh.pre = pick >= 0 ? tgt - run : -1.0;
    }
  } else if (mass) {  // rounding pushed u * Z past the total: the last sub-range with weight
    if (lane == 31 - __clz(mass)) {
      int last = -1;
      for (int q = q0; q < q1; ++q)
        if (wsum(q) > 0.f) last = q;
      sh.sub = last;
      sh.pre = -1.0;  // take its last entry with weight
    }
  }
}

// The whole block: draw inside sub-range sub ([sub * kSub, ...) of the row),
// target sh.pre measured from the sub-range start.  Thread t covers 8 entries;
// the block scan gives each warp a float target relative to its start, and the
// first thread whose range [excl, incl) holds it walks its 8 weights.  A target
// past the scanned total (rounding), or sh.pre < 0, takes the last entry with
// weight.  Returns the token (every thread).
template <bool VEC4>
__device__ int draw_in_sub(const Weights &w, int V, DrawShared &sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lo = sh.sub * kSub;
  const int hi = min(V, lo + kSub);
  const int i0 = lo + 8 * static_cast<int>(threadIdx.x);
  float v[8];
  weights8<VEC4>(w, i0, hi, v);
  float ts = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ts += v[e];
    if (v[e] > 0.f) lastpos = i0 + e;
  }
  float incl = ts;
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) sh.wsum[warp] = incl;
  if (threadIdx.x == 0) {
    sh.tidx = 0x7fffffff;
    sh.tok = -1;
  }
  __syncthreads();
  if (warp == 0) {  // per-warp float targets from a double scan of the warp totals
    const double x0 = (lane < kWarps) ? static_cast<double>(sh.wsum[lane]) : 0.0;
    double ix = x0;
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, ix, o);
      if (lane >= o) ix += y;
    }
    if (lane < kWarps) sh.trel[lane] = fmaxf(0.f, static_cast<float>(sh.pre - (ix - x0)));
  }
  // the last entry with weight in the whole sub-range (rounding fallback)
  int lp = lastpos;
  for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
  if (lane == 0 && lp >= 0) atomicMax(&sh.tok, lp);
  __syncthreads();
  const float trel = sh.trel[warp];
  if (sh.pre >= 0.0 && ts > 0.f && excl <= trel && incl > trel) atomicMin(&sh.tidx, static_cast<int>(threadIdx.x));
  __syncthreads();
  if (static_cast<int>(threadIdx.x) == sh.tidx) {
    float c = excl;
    int p = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c += v[e];
      if (p < 0 && v[e] > 0.f && c > trel) p = i0 + e;
    }
    sh.tok = (p >= 0) ? p : lastpos;  // the crossing is here; rounding: this thread's last entry with weight
  }
  __syncthreads();
  return sh.tok;
}

// One draft-token draw of a single draft row per sequence (a draft step).
// CTA (b, s) streams entries [s * kChunk, ...) of the row; warp w keeps the
// (max, sum of exp) of its sub-range s * kWarps + w.  The CTA completing the
// sequence merges the sub-range records into weights relative to the row max
// and draws.  Each lane streams its 64 entries in NR rounds (all loads of a
// round in flight) with its own running (max, sum), merged over the warp at
// the end: NR = 1 (all 64 in flight, 2 CTAs per SM) when the grid fits in two
// CTAs per SM, else NR = 2 (5 CTAs per SM at 48 registers).  Measured at vocab
// 128256: batch 32, 256 CTAs, 11 us per draw in a chain of draft steps with
// NR = 1 against 13 us with NR = 2; batch 128, 1024 CTAs, 18.7 us with NR = 2
// at 4 CTAs per SM against 20.2 us with NR = 1 and 23.8 us with NR = 4 at 32
// registers (one wave of 8 CTAs per SM, but four dependent rounds); 5 CTAs per
// SM take 0.85 us off each draw of the 4-step draft phase (1.35 waves instead
// of 1.7), 6 (40 registers, a few spilled) add 4 us.  The stream uses the default L2 policy, so
// that the completing CTA's second read of the chosen sub-range finds it in L2.
// With CLUSTER the CTAs of a row form one thread-block cluster (a row has at
// most 8 chunks): each warp stores its record into the shared memory of the
// cluster's first CTA, and after one cluster barrier that CTA draws -- no
// ticket, no round trip of the records through global memory.
template <bool VEC4, int NR, bool CLUSTER>
__global__ void __launch_bounds__(kStatThreads, NR == 1 ? 2 : 5)
    spec_draw_row_kernel(const float *__restrict__ draft, int32_t *__restrict__ draft_tokens,
                         const float *__restrict__ u, StatParams sp, float2 *__restrict__ stats,
                         float2 *__restrict__ sub, unsigned *__restrict__ tickets, unsigned *__restrict__ drawn,
                         WsHeader *hdr) {
  pdl_launch_dependents();
  {  // warm L2 with this CTA's 64 KB of the row while the previous kernel finishes (prefetch only)
    const float *x0 = draft + (static_cast<size_t>(blockIdx.x) * sp.gamma + (sp.r_begin - sp.gamma - 1)) * sp.V;
    const int lo = blockIdx.y * kChunk, hi = min(sp.V, lo + kChunk);
    for (int e = lo + 32 * static_cast<int>(threadIdx.x); e < hi; e += 32 * kStatThreads)  // one 128-byte line each
      asm volatile("prefetch.global.L2 [%0];" ::"l"(x0 + e));
  }
  pdl_wait();
  __shared__ int s_last;
  __shared__ float s_M;
  __shared__ DrawShared sh;
  __shared__ float2 s_rec[kRecSmem];
  __shared__ float2 s_wst[kWarps];  // the warps' (max, sum), merged into the chunk's statistics
  const int b = blockIdx.x, s = blockIdx.y;
  const int row = sp.r_begin - sp.gamma - 1;  // draft position
  const int V = sp.V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *x = draft + (static_cast<size_t>(b) * sp.gamma + row) * V;
  float2 *sub_b = sub + static_cast<size_t>(b) * sp.nsub;
  {
    const int g = s * kWarps + warp;
    const int lo = g * kSub, hi = min(V, lo + kSub);
    float m = -INFINITY, l = 0.f;
    if (lo < hi) {
#pragma unroll 1
      for (int h = 0; h < NR; ++h) {
        constexpr int PER = 64 / NR, F4 = PER / 4;
        float v[PER];
        if (VEC4) {
#pragma unroll
          for (int k = 0; k < F4; ++k) {
            const int i = lo + 4 * lane + 128 * (F4 * h + k);
            const float4 f = (i < hi) ? __ldg(reinterpret_cast<const float4 *>(x + i))
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            v[4 * k] = f.x, v[4 * k + 1] = f.y, v[4 * k + 2] = f.z, v[4 * k + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < PER; ++k) {
            const int i = lo + lane + 32 * (PER * h + k);
            v[k] = (i < hi) ? __ldg(x + i) : -INFINITY;
          }
        }
        float mx = v[0];
#pragma unroll
        for (int k = 1; k < PER; ++k) mx = fmaxf(mx, v[k]);
        if (mx > m) {
          l *= ex2((m - mx) * kLog2e);  // 0 while m is -inf (l is 0 then as well)
          m = mx;
        }
        if (m != -INFINITY) {  // -inf logits (masked entries) weigh 0
          const float ml = m * kLog2e;
#pragma unroll
          for (int k = 0; k < PER; ++k) l += ex2(fmaf(v[k], kLog2e, -ml));
        }
      }
    }
    for (int o = 16; o > 0; o >>= 1) {  // merge the lanes' (max, sum)
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
      const float mn = fmaxf(m, m2);
      const float mu = (mn == -INFINITY) ? 0.f : mn;
      l = l * ex2((m - mu) * kLog2e) + l2 * ex2((m2 - mu) * kLog2e);
      m = mn;
    }
    if (lane == 0) s_wst[warp] = make_float2(m, l);
    // the chunk's (max, sum of exp) of this draft row, kept for the round's rejection sample
    auto put_chunk_stats = [&] {
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_wst[w].x);
      const float Mu = (M == -INFINITY) ? 0.f : M;
      float Lt = 0.f;
      for (int w = 0; w < kWarps; ++w) Lt += s_wst[w].y * exp2f((s_wst[w].x - Mu) * kLog2e);
      stats[(static_cast<size_t>(b) * sp.nrows + sp.r_begin) * sp.nsplit + s] = make_float2(M, Lt);
    };
    if (CLUSTER) {
      if (lane == 0 && g < sp.nsub) st_cluster_f2(&s_rec[g], 0u, make_float2(m, l));
      cluster_sync_all();  // every record is in the first CTA's shared memory
      if (threadIdx.x == 32) put_chunk_stats();  // (warp 0 goes on to the pick meanwhile)
      if (s != 0) return;  // (nothing reads the other CTAs' shared memory after the barrier)
    } else {
      if (lane == 0 && g < sp.nsub) sub_b[g] = make_float2(m, l);
      __syncthreads();
      if (threadIdx.x == 32) put_chunk_stats();
      if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(&tickets[b], 1u) == static_cast<unsigned>(sp.nsplit - 1)) ? 1 : 0;
      }
      __syncthreads();
      if (!s_last) return;
      __threadfence();
    }
  }
  // this CTA completed the sequence: the sub-range records (one read, into shared memory when
  // they fit), weights relative to the row max, then the draw
  const bool rec_smem = CLUSTER || sp.nsub <= kRecSmem;
  if (!CLUSTER && rec_smem) {
    for (int q = threadIdx.x; q < sp.nsub; q += kStatThreads) s_rec[q] = __ldcg(&sub_b[q]);
    __syncthreads();
  }
  if (warp == 0) {
    auto rec = [&](int q) { return rec_smem ? s_rec[q] : __ldcg(&sub_b[q]); };
    float M = -INFINITY;
    for (int q = lane; q < sp.nsub; q += 32) M = fmaxf(M, rec(q).x);
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) s_M = M;
    auto wsum = [&](int q) {
      const float2 r = rec(q);
      return r.y * exp2f((r.x - M) * kLog2e);
    };
    pick_sub(wsum, sp.nsub, u[(static_cast<size_t>(b) * (sp.gamma + 1) + row) * 3 + 0], sh);
  }
  __syncthreads();
  int tok = -1;
  if (sh.sub >= 0) {
    const Weights w{x, nullptr, s_M, 1.f, 0.f, 0.f, 0};
    tok = draw_in_sub<VEC4>(w, V, sh);
  }
  if (threadIdx.x == 0) {
    draft_tokens[static_cast<size_t>(b) * sp.gamma + row] = tok;
    if (!CLUSTER) tickets[b] = 0u;  // left clean for the next call on this workspace
    atomicOr(&drawn[b], 1u << row);  // this row's statistics are in place
    call_check_in(hdr, sp.B, b, 0u, 0u);
  }
}

// Merge the slice statistics of unified row r into (max, 1 / sum).
__device__ __forceinline__ void merge_row(const float2 *st, int nsplit, float &M, float &iZ) {
  M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, st[s].x);
  float Z = 0.f;
  for (int s = 0; s < nsplit; ++s) Z += st[s].y * exp2f((st[s].x - M) * kLog2e);
  iZ = 1.f / Z;
}

// Rejection sampling, CTA (b, s): the acceptance decisions of sequence b (the
// same in every CTA of b), then the weight sums of the final draw over the
// sub-ranges of chunk s; the CTA completing the sequence draws and writes the
// round's tokens.  Each lane streams its 64 entries of the two rows in NR
// rounds (all loads of a round in flight): NR = 2 (32 entries of each row in
// flight, 3 CTAs per SM) when the grid fits in one wave of that, else NR = 8
// (8 of each row, held to 32 registers so that 8 CTAs share an SM: a batch of
// 128 sequences at vocab 128256 runs as one wave of 1024 CTAs).  With CLUSTER
// the CTAs of a sequence form one thread-block cluster and hand their sums to
// the first CTA's shared memory, which draws after one cluster barrier.
template <bool VEC4, int NR, bool CLUSTER>
__global__ void __launch_bounds__(kStatThreads, NR == 2 ? 3 : (NR == 4 ? 4 : 8)) spec_decide_kernel(const float *__restrict__ target,
                                                                       const float *__restrict__ draft,
                                                                       const int32_t *__restrict__ draft_tokens,
                                                                       const float *__restrict__ u, StatParams sp,
                                                                       const float2 *__restrict__ stats,
                                                                       float2 *__restrict__ sub,
                                                                       unsigned *__restrict__ tickets,
                                                                       unsigned *__restrict__ drawn,
                                                                       int32_t *__restrict__ out_tokens,
                                                                       int32_t *__restrict__ num_accepted,
                                                                       WsHeader *hdr) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float sM[33], siZ[33];
  __shared__ int s_tok[16];
  __shared__ unsigned char s_ok[16], s_bad[16];
  __shared__ int s_j, s_last, s_use_p;
  __shared__ DrawShared sh;
  __shared__ float2 s_rec[kRecSmem];
  const int b = blockIdx.x, s = blockIdx.y;
  const int g = sp.gamma, V = sp.V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the candidates' tokens and the two logits at each are loaded by warp 2 while warp 0
  // merges the row statistics (the loads do not depend on the statistics)
  constexpr int kCand = 64;  // first thread of the candidate tests (gamma <= 16, nrows <= 33)
  const int ci = static_cast<int>(threadIdx.x) - kCand;
  int xi = -1;
  bool bad = true;
  float xa = 0.f, xc = 0.f, uu = 0.f;
  if (ci >= 0 && ci < g) {
    xi = draft_tokens[static_cast<size_t>(b) * g + ci];
    bad = (xi < 0 || xi >= V);
    if (!bad) {
      xa = row_ptr(target, draft, b, ci, g, V)[xi];
      xc = row_ptr(target, draft, b, g + 1 + ci, g, V)[xi];
      uu = u[(static_cast<size_t>(b) * (g + 1) + ci) * 3 + 1];
    }
  }
  for (int r = threadIdx.x; r < sp.nrows; r += kStatThreads)
    merge_row(stats + (static_cast<size_t>(b) * sp.nrows + r) * sp.nsplit, sp.nsplit, sM[r], siZ[r]);
  __syncthreads();
  // every candidate's test at once; the chain keeps the prefix before the first rejection
  if (ci >= 0 && ci < g) {
    bool acc = false;
    if (!bad) {
      const float px = exp2f((xa - sM[ci]) * kLog2e) * siZ[ci];
      const float qx = exp2f((xc - sM[g + 1 + ci]) * kLog2e) * siZ[g + 1 + ci];
      acc = uu * qx < px;
    }
    s_tok[ci] = xi;
    s_ok[ci] = acc ? 1 : 0;
    s_bad[ci] = bad ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = g;
    for (int i = 0; i < g; ++i)
      if (s_bad[i] || !s_ok[i]) {
        j = i;
        break;
      }
    s_j = j;
  }
  __syncthreads();
  const int j = s_j;
  const int jc = g + 1 + min(j, g - 1);  // the draft row of position j (read only when j < g)
  float2 *sub_b = sub + static_cast<size_t>(b) * sp.nsub;
  {
    // the draw's weights over this warp's sub-range: the residual max(0, p - q) at a
    // rejection (and p_j as well, for the rare case where the residual sums to zero), p of
    // the bonus row otherwise; each target value serves both sums
    const float *ra = row_ptr(target, draft, b, j, g, V);
    const float *rc = row_ptr(target, draft, b, jc, g, V);
    const float Ma = sM[j], ia = siZ[j], Mc = sM[jc], ic = siZ[jc];
    const bool resid = j < g;
    const int sg = s * kWarps + warp;
    const int lo = sg * kSub, hi = min(V, lo + kSub);
    float r = 0.f, pp = 0.f;
#pragma unroll 1
    for (int h = 0; h < NR && lo < hi; ++h) {
      constexpr int PER = 64 / NR, F4 = PER / 4;
      float a[PER], c[PER];
#pragma unroll
      for (int k = 0; k < F4; ++k) {
        const int i = lo + 4 * lane + 128 * (F4 * h + k);
        if (VEC4 && i + 3 < hi) {
          const float4 fa = __ldg(reinterpret_cast<const float4 *>(ra + i));
          a[4 * k] = fa.x, a[4 * k + 1] = fa.y, a[4 * k + 2] = fa.z, a[4 * k + 3] = fa.w;
          const float4 fc = resid ? __ldg(reinterpret_cast<const float4 *>(rc + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
          c[4 * k] = fc.x, c[4 * k + 1] = fc.y, c[4 * k + 2] = fc.z, c[4 * k + 3] = fc.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a[4 * k + e] = (i + e < hi) ? __ldg(ra + i + e) : -INFINITY;
            c[4 * k + e] = (resid && i + e < hi) ? __ldg(rc + i + e) : 0.f;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const float pa = exp2f((a[e] - Ma) * kLog2e) * ia;  // p, as the weights functions compute it
        pp += pa;
        r += resid ? fmaxf(0.f, pa - exp2f((c[e] - Mc) * kLog2e) * ic) : pa;
      }
    }
    r = warp_sum_xor(r, 1, 16);
    pp = warp_sum_xor(pp, 1, 16);
    if (CLUSTER) {
      if (lane == 0 && sg < sp.nsub) st_cluster_f2(&s_rec[sg], 0u, make_float2(r, pp));
      cluster_sync_all();  // every sum is in the first CTA's shared memory
      if (s != 0) return;  // (nothing reads the other CTAs' shared memory after the barrier)
    } else {
      if (lane == 0 && sg < sp.nsub) sub_b[sg] = make_float2(r, pp);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(&tickets[b], 1u) == static_cast<unsigned>(sp.nsplit - 1)) ? 1 : 0;
      }
      __syncthreads();
      if (!s_last) return;
      __threadfence();
    }
  }
  // this CTA completed the sequence: the sub-range sums (one read, into shared memory when
  // they fit), then the draw of the correction (or bonus) token
  const bool rec_smem = CLUSTER || sp.nsub <= kRecSmem;
  if (!CLUSTER && rec_smem) {
    for (int q = threadIdx.x; q < sp.nsub; q += kStatThreads) s_rec[q] = __ldcg(&sub_b[q]);
    __syncthreads();
  }
  if (warp == 0) {
    auto rec = [&](int q) { return rec_smem ? s_rec[q] : __ldcg(&sub_b[q]); };
    float zr = 0.f;
    for (int q = lane; q < sp.nsub; q += 32) zr += rec(q).x;
    zr = warp_sum_xor(zr, 1, 16);
    const int use_p = (j < g && !(zr > 0.f)) ? 1 : 0;  // the residual vanished through rounding: draw from p_j
    if (lane == 0) s_use_p = use_p;
    auto wsum = [&](int q) { return use_p ? rec(q).y : rec(q).x; };
    pick_sub(wsum, sp.nsub, u[(static_cast<size_t>(b) * (g + 1) + j) * 3 + 2], sh);
  }
  __syncthreads();
  int tok = -1;
  if (sh.sub >= 0) {
    const Weights wr{row_ptr(target, draft, b, j, g, V), row_ptr(target, draft, b, jc, g, V), sM[j], siZ[j],
                     sM[jc], siZ[jc], (j < g && !s_use_p) ? 1 : 0};
    tok = draw_in_sub<VEC4>(wr, V, sh);
  }
  if (threadIdx.x == 0) {
    int32_t *o = out_tokens + static_cast<size_t>(b) * (g + 1);
    for (int i = 0; i < j; ++i) o[i] = s_tok[i];
    o[j] = tok;
    for (int i = j + 1; i <= g; ++i) o[i] = -1;
    num_accepted[b] = j;
    if (j < g && s_bad[j]) raise_error_sr(hdr, 0x4u);
    if (!CLUSTER) tickets[b] = 0u;
    // the draws' marks go back to zero with every rejection sample; reusing their statistics
    // needs all gamma of them
    const unsigned have = drawn[b];
    drawn[b] = 0u;
    if (sp.reuse && have != (1u << g) - 1u) raise_error_sr(hdr, 0x40u);
    call_check_in(hdr, sp.B, b, 0u, 0u);
  }
}

}  // namespace

SpecPlan plan_spec(int B, int gamma, int V) {
  SpecPlan p{};
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.split = kChunk;
  p.nsplit = (V + p.split - 1) / p.split;
  p.nsub = (V + kSub - 1) / kSub;
  p.nrows = 2 * gamma + 1;
  p.off_tickets = kAlign;
  p.off_drawn = align_up(p.off_tickets + sizeof(unsigned) * static_cast<size_t>(B));
  p.off_stats = align_up(p.off_drawn + sizeof(unsigned) * static_cast<size_t>(B));
  p.off_sub = align_up(p.off_stats + sizeof(float2) * static_cast<size_t>(B) * p.nrows * p.nsplit);
  p.ws_bytes = align_up(p.off_sub + sizeof(float2) * static_cast<size_t>(B) * p.nsub);
  return p;
}

// Resident CTAs of kStatThreads threads per SM for a kernel (0 if the query fails).
static int ctas_per_sm(const void *fn) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kStatThreads, 0) != cudaSuccess) n = 0;
  return n;
}

cudaError_t launch_spec(const SpecPlan &p, const SpecArgs &a) {
  StatParams sp;
  sp.reuse = 0;
  sp.B = p.B;
  sp.gamma = p.gamma;
  sp.V = p.V;
  sp.split = p.split;
  sp.nsplit = p.nsplit;
  sp.nrows = p.nrows;
  sp.nsub = p.nsub;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  unsigned *tickets = reinterpret_cast<unsigned *>(ws + p.off_tickets);
  unsigned *drawn = reinterpret_cast<unsigned *>(ws + p.off_drawn);
  float2 *stats = reinterpret_cast<float2 *>(ws + p.off_stats);
  float2 *sub = reinterpret_cast<float2 *>(ws + p.off_sub);
  WsHeader *hdr = static_cast<WsHeader *>(a.ws);
  const bool vec4 = (p.V % 4) == 0 && (reinterpret_cast<uintptr_t>(a.draft) % 16) == 0 &&
                    (a.target == nullptr || (reinterpret_cast<uintptr_t>(a.target) % 16) == 0);
  const dim3 grid(p.B, p.nsplit);
  // the round counts that keep every CTA of the grid resident at once when the grid is small
  const long long ctas = static_cast<long long>(p.B) * p.nsplit, sms = current_sm_count();
  static const int occ_draw1 = ctas_per_sm(reinterpret_cast<const void *>(spec_draw_row_kernel<true, 1, false>));
  static const int occ_decide2 = ctas_per_sm(reinterpret_cast<const void *>(spec_decide_kernel<true, 2, false>));
  if (a.mode == 1) {  // draft draws: one launch per drawn row
    const bool one = ctas <= occ_draw1 * sms;
    // a row of at most 8 chunks (vocab up to 131072) draws inside one cluster
    const bool cl = p.nsplit <= 8;
    auto kd = cl ? (vec4 ? (one ? spec_draw_row_kernel<true, 1, true> : spec_draw_row_kernel<true, 2, true>)
                         : (one ? spec_draw_row_kernel<false, 1, true> : spec_draw_row_kernel<false, 2, true>))
                 : (vec4 ? (one ? spec_draw_row_kernel<true, 1, false> : spec_draw_row_kernel<true, 2, false>)
                         : (one ? spec_draw_row_kernel<false, 1, false> : spec_draw_row_kernel<false, 2, false>));
    const int r0 = a.row < 0 ? 0 : a.row, r1 = a.row < 0 ? p.gamma : a.row + 1;
    for (int r = r0; r < r1; ++r) {
      sp.r_begin = p.gamma + 1 + r;
      sp.nr = 1;
      const cudaError_t e =
          cl ? launch_pdl_cluster(kd, grid, dim3(kStatThreads), dim3(1, p.nsplit, 1), 0, a.stream, a.draft,
                                  a.draft_tokens, a.u, sp, stats, sub, tickets, drawn, hdr)
             : launch_pdl(kd, grid, dim3(kStatThreads), 0, a.stream, a.draft, a.draft_tokens, a.u, sp, stats, sub,
                          tickets, drawn, hdr);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  // MGD_VERIFY_DRAWN: the gamma draft rows' statistics were left by this round's draws, so
  // only the gamma + 1 target rows are streamed here
  sp.reuse = a.mode == 2 ? 1 : 0;
  sp.r_begin = 0;
  sp.nr = sp.reuse ? p.gamma + 1 : p.nrows;
  const dim3 g1(p.B * sp.nr, p.nsplit);
  cudaError_t e = launch_pdl(vec4 ? spec_stats_kernel<true> : spec_stats_kernel<false>, g1, dim3(kStatThreads), 0,
                             a.stream, a.target, a.draft, sp, stats);
  if (e != cudaSuccess) return e;
  const bool wide = ctas <= occ_decide2 * sms;
  const bool cl = p.nsplit <= 8;  // a sequence of at most 8 chunks decides inside one cluster
  auto kc = cl ? (vec4 ? (wide ? spec_decide_kernel<true, 2, true> : spec_decide_kernel<true, 8, true>)
                       : (wide ? spec_decide_kernel<false, 2, true> : spec_decide_kernel<false, 8, true>))
               : (vec4 ? (wide ? spec_decide_kernel<true, 2, false> : spec_decide_kernel<true, 8, false>)
                       : (wide ? spec_decide_kernel<false, 2, false> : spec_decide_kernel<false, 8, false>));
  if (cl)
    return launch_pdl_cluster(kc, grid, dim3(kStatThreads), dim3(1, p.nsplit, 1), 0, a.stream, a.target, a.draft,
                              a.draft_tokens, a.u, sp, stats, sub, tickets, drawn, a.out_tokens, a.num_accepted,
                              hdr);
  return launch_pdl(kc, grid, dim3(kStatThreads), 0, a.stream,
                    a.target, a.draft, a.draft_tokens, a.u, sp, stats, sub, tickets, drawn, a.out_tokens,
                    a.num_accepted, hdr);
}

}  // namespace mgd
