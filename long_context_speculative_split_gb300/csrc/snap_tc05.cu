// SnapKV window scores on the 5th-generation tensor cores (tcgen05 + TMEM),
// both passes in one persistent kernel that streams K from HBM once.
//
// MagicDec notes, section 4.4 (SnapKV as the static selector) and appendix A.1
// (selection at prefill).  Step 1 of the selection (see snapkv.cu): the W
// window queries of a KV head (W * G = 128 rows) attend causally over the
// context; pass 1 gets each row's log-sum-exp, pass 2 sums each prefix key's
// probabilities over the 128 rows.  Both passes are dense contractions
// (2 * 128 * D flop per key), so they run as tcgen05.mma with M = N = 128:
//
//   pass 1: S  = Qw K^T   (TMEM lane = window row, column = key): every thread
//           owns one row and keeps its own online max / sum -- no shuffles;
//   pass 2: S^T = K Qw^T  (TMEM lane = key, column = window row): every thread
//           owns one key and sums exp2(s - lse_row) over the rows in registers.
//
// One read of K.  The work is cut into slices of p.C keys (1536, longer for
// capacities above 64 such slices) of one (sequence, KV head) pair.  A CTA
// runs pass 1 over a slice, publishes the slice's per-row (max, sum) and
// counts it in the pair's counter, waits until every slice of the pair has
// done the same (they were claimed at nearly the same moment by other CTAs,
// since slices are handed out in order from one atomic counter), merges the
// partials into the rows' log-sum-exp, and then runs pass 2 over the same
// slice.  Between the two reads of a tile the whole GPU fetches only about one
// slice per CTA from HBM, so most second reads come from L2 instead of HBM.
//
// Progress, whatever the residency: the global counter hands out tickets of a
// pair, and each ticket claims the pair's next unclaimed slice from a per-pair
// counter.  Before a CTA waits for its pair, it claims and runs pass 1 over
// every slice of the pair that nobody has claimed yet (help first); so it
// waits only for slices that running CTAs hold.  A CTA claims a new pair only
// after its current pair's exchange completed, and nothing between claiming a
// slice and publishing it waits on another CTA: the waits always end, even
// when only a few CTAs are resident (another kernel holding SMs).  In the
// usual case every slice is claimed long before its pair's first CTA is done
// with pass 1, and helping never happens.  Every wait is bounded
// (kWaitLimitNs) and raises MGD_DEVERR_TIMEOUT instead of hanging.
//
// L2: pass-1 tile loads carry an evict_last hint and pass-2 loads (the last
// read) evict_first, so the slices between their two reads (one per CTA)
// keep their place against the rest of the stream.
//
// CTA = 10 warps, 2 CTAs per SM: warp 0 claims slices and issues TMA (the 128
// window rows of the pair, then its 128-key K tiles -- pass 1's, then the same
// tiles again for pass 2 -- into a 2-stage ring) and describes the work to the
// other roles as a stream of segments (pass 1 of a slice, the pair's exchange,
// pass 2 of a slice) through a small shared-memory ring; warp 1 owns the TMEM
// allocation and one thread issues the MMAs (8 k-steps of K = 16 per tile)
// into a double-buffered 2 x 128-column fp32 accumulator, warps 2..9 drain it
// (tcgen05.ld) as two groups of 4 warps taking alternate tiles, one warp per
// TMEM lane quadrant, and do the exchange.  Operands are K-major bf16 with
// 128-byte swizzling, exactly the layout TMA writes.  Used when W * G == 128
// and D == 128 (the Llama-3.1-8B shape with a 32-row window); other shapes use
// the kernels in snapkv.cu.
#include <algorithm>

#include "common.cuh"

namespace mgd {
namespace {

constexpr int kT5Keys = 128;
constexpr int kT5Groups = 2;                // softmax groups of 4 warps, one TMEM accumulator each
constexpr int kT5Stages = 2;                // K tiles in flight
constexpr int kT5CtasPerSm = 2;
constexpr int kT5SoftWarps = 4 * kT5Groups;
constexpr int kT5Threads = 64 + 32 * kT5SoftWarps;
constexpr int kT5Half = 128 * 128;          // one 64-column (128 B) atom column of 128 rows
constexpr int kT5TileBytes = 2 * kT5Half;   // 128 rows x 128 bf16
constexpr uint32_t kT5TmemCols = 128 * kT5Groups;  // one 128-column accumulator per group
static_assert(kT5Groups == 2 || kT5Groups == 4, "tcgen05.alloc takes a power-of-two column count");
constexpr int kExchThread = 64;             // first softmax thread: segment broadcast and exchange
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRing = 8;                    // segment messages in flight between the producer and its consumers

constexpr uint32_t kIdescM128N128 = umma_idesc_bf16(128, 128);

// Segment kinds.  Flags: kFirst -- the first segment of a pair (the MMA thread
// waits for the pair's window rows); kLast -- the last (it then releases them).
enum : int { kSegP1 = 0, kSegXchg = 1, kSegP2 = 2, kSegEnd = 3 };
constexpr int kFirst = 1, kLast = 2;

struct T5Layout {
  static constexpr int off_q = 0;                                   // 32 KB window rows
  static constexpr int off_k = kT5TileBytes;                        // kT5Stages x 32 KB
  static constexpr int off_bar = off_k + kT5Stages * kT5TileBytes;  // 32 mbarriers
  static constexpr int off_tmem = off_bar + 32 * 8;
  static constexpr int off_ring = off_tmem + 16;                    // int4 [kRing] segments
  static constexpr int off_bcast = off_ring + kRing * 16;           // int4 [2] softmax broadcast
  static constexpr int off_abort = off_bcast + 2 * 16;              // int
  static constexpr int off_lse = off_abort + 16;                    // float [128]
  static constexpr int off_red = off_lse + 128 * 4;                 // float [groups][2][128]
  static constexpr int bytes = off_red + kT5Groups * 2 * 128 * 4;
  static constexpr int alloc = bytes + 1024;
};

struct T5Params {
  int W, G, Hkv, C, nslice, kv_cap, units;  // C: keys per slice; units = pairs * nslice tickets
  float sl2;
  size_t off_cnt, off_part, off_scores;
};

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Slice `slice` (p.C keys from `start`) of pair `pair` = (sequence b, KV head
// hkv).  nt1 / nt2 = 128-key tiles of pass 1 (keys < L) and pass 2 (prefix
// keys < L - W); ns = slices of the pair that hold pass-1 keys.
struct Slice {
  int b, hkv, L, start, end2, nt1, nt2, ns;
  bool valid;
};
__device__ __forceinline__ Slice slice_of(int pair, int slice, const int32_t *__restrict__ kv_len,
                                          const T5Params &p) {
  Slice j;
  j.b = pair / p.Hkv;
  j.hkv = pair - j.b * p.Hkv;
  j.L = kv_len[j.b];
  j.valid = j.L >= p.W && j.L <= p.kv_cap;
  j.start = slice * p.C;
  const int end1 = min(j.start + p.C, j.L);
  j.end2 = min(j.start + p.C, j.L - p.W);
  j.nt1 = (j.valid && end1 > j.start) ? (end1 - j.start + kT5Keys - 1) / kT5Keys : 0;
  j.nt2 = (j.valid && j.end2 > j.start) ? (j.end2 - j.start + kT5Keys - 1) / kT5Keys : 0;
  j.ns = j.valid ? (j.L + p.C - 1) / p.C : 0;
  return j;
}

// Pass 1 on one accumulator tile: window row tl against keys kt0 .. kt0+127
// (keys after `pos`, the row's last visible key, masked when the tile reaches
// the window at `wstart`), folded into the row's running (max, sum) in the
// exp2 domain.  Hands the accumulator back once both halves are in registers.
__device__ __forceinline__ void pass1_tile(uint32_t lane_addr, int kt0, int wstart, int pos, float sl2,
                                           uint64_t *acc_empty, int lane, float &m_run, float &l_run) {
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float v[2][32];
    tmem_ld32(lane_addr + h * 64, v[0]);
    tmem_ld32(lane_addr + h * 64 + 32, v[1]);
    if (h == 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
    if (kt0 + kT5Keys - 1 > wstart) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (kt0 + 64 * h + 32 * i + c > pos) v[i][c] = -INFINITY;
    }
    // the 64 values as 32 pairs: four 3-input max chains, then paired (f32x2)
    // scale-and-shift and sums, two exponentials per pair
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 32; ++j) mx[j & 3] = fmax3(mx[j & 3], v[j >> 4][(j & 15) * 2], v[j >> 4][(j & 15) * 2 + 1]);
    const float mn = fmaxf(m_run, fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * sl2);  // sl2 > 0
    const float mu = (mn == -INFINITY) ? 0.f : mn;
    const float2 s2 = make_float2(sl2, sl2), nm = make_float2(-mu, -mu);
    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 x = __ffma2_rn(make_float2(v[j >> 4][(j & 15) * 2], v[j >> 4][(j & 15) * 2 + 1]), s2, nm);
      acc[j & 1] = __fadd2_rn(acc[j & 1], make_float2(ex2(x.x), ex2(x.y)));
    }
    l_run = l_run * ex2(m_run - mu) + ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y));
    m_run = mn;
  }
}

// Pass 2 on one accumulator tile: key tl against the 128 window rows; returns
// sum over rows of exp2(s * sl2 - lse_row), with -lse in shared memory.
__device__ __forceinline__ float pass2_tile(uint32_t lane_addr, const float *sm_nlse, float sl2, uint64_t *acc_empty,
                                            int lane) {
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 s2 = make_float2(sl2, sl2);
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float v[2][32];
    tmem_ld32(lane_addr + h * 64, v[0]);
    tmem_ld32(lane_addr + h * 64 + 32, v[1]);
    if (h == 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 nl = *reinterpret_cast<const float4 *>(&sm_nlse[64 * h + 32 * i + c]);
        const float2 x0 = __ffma2_rn(make_float2(v[i][c], v[i][c + 1]), s2, make_float2(nl.x, nl.y));
        const float2 x1 = __ffma2_rn(make_float2(v[i][c + 2], v[i][c + 3]), s2, make_float2(nl.z, nl.w));
        acc[0] = __fadd2_rn(acc[0], make_float2(ex2(x0.x), ex2(x0.y)));
        acc[1] = __fadd2_rn(acc[1], make_float2(ex2(x1.x), ex2(x1.y)));
      }
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

// Segment slots are volatile shared memory, written and read one field at a time.
__device__ __forceinline__ void put_seg(volatile int4 *d, int a, int b, int c, int e) {
  d->x = a;
  d->y = b;
  d->z = c;
  d->w = e;
}
__device__ __forceinline__ int4 get_seg(const volatile int4 *d) { return make_int4(d->x, d->y, d->z, d->w); }

// A bounded wait that also gives up at once after any other wait of the CTA
// gave up; a failure raises the timeout bit and sets the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, WsHeader *hdr,
                                              volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  raise_error_sr(hdr, 0x8u);
  *abort_flag = 1;
  return false;
}

__global__ void __launch_bounds__(kT5Threads, kT5CtasPerSm)
    snap_score_fused(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                     const int32_t *__restrict__ kv_len, unsigned char *__restrict__ ws, T5Params p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T5Layout::off_bar);
  uint64_t *q_full = bars + 0;      // window rows of the pair landed
  uint64_t *q_empty = bars + 1;     // every MMA of the previous pair done: the rows may be replaced
  uint64_t *full = bars + 2;                    // [kT5Stages] K tile landed
  uint64_t *empty = full + kT5Stages;           // [kT5Stages] K tile consumed by its MMAs
  uint64_t *acc_full = empty + kT5Stages;       // [kT5Groups] accumulator written
  uint64_t *acc_empty = acc_full + kT5Groups;   // [kT5Groups] accumulator drained by its group
  uint64_t *seg_full = acc_empty + kT5Groups;   // [kRing] segment slot written
  uint64_t *seg_empty = seg_full + kRing;       // [kRing] segment slot read by the MMA thread and the softmax warps
  uint64_t *xchg = seg_empty + kRing;           // this pair's exchange is complete (the producer may claim the next pair)
  uint64_t *mma_done = xchg + 1;                // final: every MMA issued has completed
  static_assert(2 + 2 * kT5Stages + 2 * kT5Groups + 2 * kRing + 2 <= 32, "mbarrier slots");
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + T5Layout::off_tmem);
  volatile int4 *ring = reinterpret_cast<volatile int4 *>(smem + T5Layout::off_ring);
  // the exchange thread's copy of each segment for the softmax warps, double-buffered so that
  // a slot is rewritten only after every thread passed the next segment's barrier
  volatile int4 *bcast = reinterpret_cast<volatile int4 *>(smem + T5Layout::off_bcast);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + T5Layout::off_abort);
  float *sm_nlse = reinterpret_cast<float *>(smem + T5Layout::off_lse);  // minus each row's log2-sum-exp
  float *sm_red = reinterpret_cast<float *>(smem + T5Layout::off_red);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  const int pairs = p.units / p.nslice;
  unsigned *cnt = reinterpret_cast<unsigned *>(ws + p.off_cnt);  // [pairs] slices published
  unsigned *claim = cnt + pairs;                                  // [pairs] slices claimed
  float2 *part = reinterpret_cast<float2 *>(ws + p.off_part);    // [pairs][nslice][128] (max, sum)
  float *scores = reinterpret_cast<float *>(ws + p.off_scores);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kT5Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kT5Groups; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);  // the 4 warps of the group draining buffer a
    }
    for (int a = 0; a < kRing; ++a) {
      mbar_init(&seg_full[a], 1);
      mbar_init(&seg_empty[a], 2);  // the MMA thread and the exchange thread
    }
    mbar_init(xchg, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // the whole warp allocates the accumulator columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kT5TmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ claims, segments, TMA
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&qmap);
      // pass-1 tiles stay in L2 for their second read; pass-2 reads are the last
      const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
      int stage = 0, qn = 0, msg = 0, groups = 0;
      uint32_t phase = 0;
      int issued = 0;  // K tiles issued; tile i went to stage i % kT5Stages in phase i / kT5Stages
      unsigned tickets = 0;  // successful claims from the header's work counter
      bool ok = true;
      auto emit = [&](int pair, int slice, int kind, int flags) {
        const int slot = msg % kRing;
        if (!wait_or_abort(&seg_empty[slot], ((msg / kRing) & 1u) ^ 1u, hdr, abort_flag)) return false;
        put_seg(&ring[slot], pair, slice, kind, flags);
        mbar_arrive(&seg_full[slot]);
        ++msg;
        return true;
      };
      // the K tiles of one pass over one slice (and the pair's window rows after the
      // first tiles of its first slice, so their HBM latency overlaps the previous pair)
      auto tiles = [&](const Slice &jb, bool pass1, bool with_q) {
        const int nt = pass1 ? jb.nt1 : jb.nt2;
        for (int i = 0; i <= nt; ++i) {
          if (with_q && i == min(nt, kT5Stages)) {
            if (!wait_or_abort(q_empty, (qn & 1u) ^ 1u, hdr, abort_flag)) return false;
            mbar_arrive_expect_tx(q_full, kT5TileBytes);
            for (int h = 0; h < 2; ++h)
              tma_load_4d(smem + T5Layout::off_q + h * kT5Half, &qmap, q_full, 64 * h, jb.hkv * p.G, 0, jb.b);
            ++qn;
          }
          if (i == nt) break;
          if (!wait_or_abort(&empty[stage], phase ^ 1u, hdr, abort_flag)) return false;
          mbar_arrive_expect_tx(&full[stage], kT5TileBytes);
          unsigned char *st = smem + T5Layout::off_k + stage * kT5TileBytes;
          const int key0 = jb.start + i * kT5Keys;
          for (int h = 0; h < 2; ++h)  // two boxes of 64 columns x 128 keys (16 KB each)
            tma_load_4d_hint(st + h * kT5Half, &kmap, &full[stage], 64 * h, key0, jb.hkv, jb.b, pass1 ? keep : drop);
          ++issued;
          if (++stage == kT5Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      while (ok) {
        // the previous pair's exchange is complete before a new pair is claimed
        if (groups > 0 && !wait_or_abort(xchg, (groups - 1) & 1u, hdr, abort_flag)) break;
        // a ticket of a pair from the global counter, then the pair's next unclaimed slice
        int pair = -1, s0 = -1;
        Slice jb{};
        while (true) {
          const unsigned u = atomicAdd(&hdr->next_unit, 1u);
          if (u >= static_cast<unsigned>(p.units)) break;
          ++tickets;
          const int pr = static_cast<int>(u) / p.nslice, ticket = static_cast<int>(u) - pr * p.nslice;
          jb = slice_of(pr, 0, kv_len, p);
          if (!jb.valid) {
            if (ticket == 0 && jb.hkv == 0) raise_error_sr(hdr, 0x2u);
            continue;
          }
          if (ticket >= jb.ns) continue;  // a pair has as many tickets as slices
          const unsigned s = atomicAdd(&claim[pr], 1u);
          if (s < static_cast<unsigned>(jb.ns)) {
            pair = pr;
            s0 = static_cast<int>(s);
            break;
          }  // else a helper already took every slice of this pair
        }
        if (pair < 0) break;
        // pass 1 over the claimed slice, then over every slice of the pair nobody has claimed yet
        uint64_t held = 0;
        bool first = true;
        for (int cur = s0;;) {
          held |= 1ull << cur;
          const Slice sl = slice_of(pair, cur, kv_len, p);
          if (!(ok = emit(pair, cur, kSegP1, first ? kFirst : 0)) || !(ok = tiles(sl, true, first))) break;
          first = false;
          if (ld_acquire_gpu(&claim[pair]) >= static_cast<unsigned>(jb.ns)) break;
          const unsigned s = atomicAdd(&claim[pair], 1u);
          if (s >= static_cast<unsigned>(jb.ns)) break;
          cur = static_cast<int>(s);
        }
        if (!ok) break;
        // the exchange, then pass 2 over the held slices that have prefix keys
        int last2 = -1;
        for (int s = 0; s < jb.ns; ++s)
          if (((held >> s) & 1ull) && slice_of(pair, s, kv_len, p).nt2 > 0) last2 = s;
        if (!(ok = emit(pair, jb.ns, kSegXchg, last2 < 0 ? kLast : 0))) break;
        for (int s = 0; s <= last2 && ok; ++s) {
          if (!((held >> s) & 1ull)) continue;
          const Slice sl = slice_of(pair, s, kv_len, p);
          if (sl.nt2 == 0) continue;
          ok = emit(pair, s, kSegP2, s == last2 ? kLast : 0) && tiles(sl, false, false);
        }
        ++groups;
      }
      if (ok) emit(-1, 0, kSegEnd, 0);
      // the selection kernel that follows checks the sum against the number of tickets
      if (tickets) atomicAdd(&hdr->claimed, tickets);
      // every copy this thread issued has landed before the CTA moves on
      for (int s = 0; s < kT5Stages && s < issued; ++s) {
        const int last = s + kT5Stages * ((issued - 1 - s) / kT5Stages);  // the stage's last tile
        mbar_wait(&full[s], static_cast<uint32_t>(last / kT5Stages) & 1u);
      }
      if (qn > 0) mbar_wait(q_full, static_cast<uint32_t>(qn - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_addr(smem + T5Layout::off_q);
      int stage = 0, qn = 0;
      uint32_t used = 0;  // bit a: parity of the tiles written into accumulator buffer a so far
      uint32_t phase = 0;
      for (int msg = 0;; ++msg) {
        const int slot = msg % kRing;
        if (!wait_or_abort(&seg_full[slot], (msg / kRing) & 1u, hdr, abort_flag)) break;
        const int4 sg = get_seg(&ring[slot]);
        mbar_arrive(&seg_empty[slot]);
        if (sg.z == kSegEnd) break;
        if (sg.z != kSegXchg) {
          if (sg.w & kFirst) {
            if (!wait_or_abort(q_full, qn & 1u, hdr, abort_flag)) break;
            ++qn;
          }
          const Slice jb = slice_of(sg.x, sg.y, kv_len, p);
          const bool p1 = sg.z == kSegP1;
          const int nt = p1 ? jb.nt1 : jb.nt2;
          bool ok = true;
          for (int i = 0; i < nt; ++i) {
            // tile i of a segment always goes to buffer (and softmax group) i % kT5Groups, so a
            // slice's arithmetic does not depend on what the CTA processed before it
            const int a = i % kT5Groups;
            if (!wait_or_abort(&full[stage], phase, hdr, abort_flag) ||
                !wait_or_abort(&acc_empty[a], ((used >> a) & 1u) ^ 1u, hdr, abort_flag)) {
              ok = false;
              break;
            }
            used ^= 1u << a;
            tc_fence_after();
            const uint32_t k_base = smem_addr(smem + T5Layout::off_k + stage * kT5TileBytes);
            const uint32_t a_base = p1 ? q_base : k_base;
            const uint32_t b_base = p1 ? k_base : q_base;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kT5Half + (kk & 3) * 32;
              umma_f16(tmem + a * 128, umma_desc(a_base + off), umma_desc(b_base + off), kIdescM128N128,
                       kk > 0 ? 1u : 0u);
            }
            umma_commit(&empty[stage]);
            umma_commit(&acc_full[a]);
            if (++stage == kT5Stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
        }
        if (sg.w & kLast) umma_commit(q_empty);
      }
      umma_commit(mma_done);  // arrives once every MMA issued above has completed
      mbar_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    // kT5Groups groups of 4 warps take each segment's tiles round robin (tile i
    // goes to group i % kT5Groups, which drains accumulator buffer
    // i % kT5Groups); warp w of a group reads TMEM lane quadrant
    // w % 4, all 128 columns of its lane, in two halves of 64.  All softmax
    // threads take the same path through the segment stream, so the named
    // barriers below always see every one of them.
    const int qd = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int tl = qd * 32 + lane;  // this thread's TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(qd * 32) << 16) + grp * 128;
    const bool exch = threadIdx.x == kExchThread;
    uint32_t drained = 0;  // tiles this group has drained so far (the parity of its buffer's phase)
    for (int msg = 0;; ++msg) {
      if (exch) {
        const int slot = msg % kRing;
        const bool got = wait_or_abort(&seg_full[slot], (msg / kRing) & 1u, hdr, abort_flag);
        const int4 g = got ? get_seg(&ring[slot]) : make_int4(-1, 0, kSegEnd, 0);
        put_seg(&bcast[msg & 1], g.x, g.y, g.z, g.w);
        mbar_arrive(&seg_empty[slot]);
      }
      named_bar(1, kT5SoftWarps * 32);
      const int4 sg = get_seg(&bcast[msg & 1]);
      if (sg.z == kSegEnd) break;
      const int pair = sg.x;
      if (sg.z == kSegP1) {
        // ---- pass 1 over one slice, its partial published for the pair's exchange
        const Slice jb = slice_of(pair, sg.y, kv_len, p);
        float m_run = -INFINITY, l_run = 0.f;
        const int pos = jb.L - p.W + tl / p.G;  // last key visible to window row tl
#pragma unroll 1
        for (int i = grp; i < jb.nt1; i += kT5Groups) {
          // the accumulator reads are warp-collective: a warp skips a tile only as a whole
          if (!__all_sync(0xffffffffu, wait_or_abort(&acc_full[grp], drained++ & 1u, hdr, abort_flag))) continue;
          tc_fence_after();
          pass1_tile(lane_addr, jb.start + i * kT5Keys, jb.L - p.W, pos, p.sl2, &acc_empty[grp], lane, m_run, l_run);
        }
        // combine the groups' (max, sum) of each row into the slice's partial and publish it
        if (grp > 0) {
          sm_red[grp * 256 + tl] = m_run;
          sm_red[grp * 256 + 128 + tl] = l_run;
        }
        named_bar(1, kT5SoftWarps * 32);
        if (grp == 0) {
          float mn = m_run;
#pragma unroll
          for (int g = 1; g < kT5Groups; ++g) mn = fmaxf(mn, sm_red[g * 256 + tl]);
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          float l = l_run * exp2f(m_run - mu);
#pragma unroll
          for (int g = 1; g < kT5Groups; ++g) l += sm_red[g * 256 + 128 + tl] * exp2f(sm_red[g * 256 + tl] - mu);
          part[(static_cast<size_t>(pair) * p.nslice + sg.y) * 128 + tl] = make_float2(mn, l);
        }
        named_bar(1, kT5SoftWarps * 32);
        if (exch) {  // after the barrier, one fence orders the 128 rows written above before the count
          __threadfence();
          atomicAdd(&cnt[pair], 1u);
        }
      } else if (sg.z == kSegXchg) {
        // ---- wait for every slice of the pair (sg.y of them), then merge their partials into -lse
        const int ns = sg.y;
        if (exch && !*abort_flag && !spin_until_geq(&cnt[pair], static_cast<unsigned>(ns))) {
          raise_error_sr(hdr, 0x8u);
          *abort_flag = 1;
        }
        named_bar(1, kT5SoftWarps * 32);
        if (grp == 0) {  // merge the partials of every slice of row tl
          const float2 *pp = part + static_cast<size_t>(pair) * p.nslice * 128 + tl;
          float M = -INFINITY, S = 0.f;
          for (int s0 = 0; s0 < ns; s0 += 8) {
            float2 x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = (s0 + k < ns) ? __ldcg(pp + (s0 + k) * 128) : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (!(x[k].y > 0.f)) continue;
              const float mn = fmaxf(M, x[k].x);
              S = S * exp2f(M - mn) + x[k].y * exp2f(x[k].x - mn);
              M = mn;
            }
          }
          sm_nlse[tl] = -(M + log2f(S));
        }
        named_bar(1, kT5SoftWarps * 32);
        if (exch) mbar_arrive(xchg);
      } else {
        // ---- pass 2 over one slice (its tiles now mostly come from L2)
        const Slice jb = slice_of(pair, sg.y, kv_len, p);
        float *srow = scores + static_cast<size_t>(pair) * p.kv_cap;
#pragma unroll 1
        for (int i = grp; i < jb.nt2; i += kT5Groups) {
          if (!__all_sync(0xffffffffu, wait_or_abort(&acc_full[grp], drained++ & 1u, hdr, abort_flag))) continue;
          tc_fence_after();
          const float sc = pass2_tile(lane_addr, sm_nlse, p.sl2, &acc_empty[grp], lane);
          const int key = jb.start + i * kT5Keys + tl;
          if (key < jb.end2) srow[key] = sc;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kT5TmemCols) : "memory");
  }
}

}  // namespace

bool snap_tc05_eligible(const SnapPlan &p) {
  return p.D == 128 && p.rows == 128 && p.RG == 1 && p.C % kT5Keys == 0 && p.nchunk <= kSnapMaxSlices;
}

cudaError_t launch_snap_score_tc05(const SnapPlan &pl, const SnapArgs &a, const CUtensorMap &kmap,
                                   const CUtensorMap &qmap) {
  T5Params kp;
  kp.W = pl.W;
  kp.G = pl.G;
  kp.Hkv = pl.Hkv;
  kp.C = pl.C;
  kp.nslice = pl.nchunk;
  kp.kv_cap = pl.kv_cap;
  kp.units = pl.pairs * pl.nchunk;
  kp.sl2 = a.sm_scale * kLog2e;
  kp.off_cnt = pl.off_cnt;
  kp.off_part = pl.off_part;
  kp.off_scores = pl.off_scores;
  auto kern = snap_score_fused;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T5Layout::alloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // persistent grid: two CTAs per SM (what the kernel's registers and shared
  // memory allow); a CTA that only starts after others finished finds no job
  const int grid = std::min(kp.units, kT5CtasPerSm * current_sm_count());
  return launch_pdl(kern, dim3(grid), dim3(kT5Threads), T5Layout::alloc, a.stream, kmap, qmap, a.kv_len,
                    static_cast<unsigned char *>(a.ws), kp);
}

}  // namespace mgd
