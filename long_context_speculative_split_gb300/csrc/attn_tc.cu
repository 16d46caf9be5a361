// Split-KV ("flash-decoding") GQA attention for the verify and draft passes,
// bf16 K/V/Q, float32 softmax and accumulation, sm_103a.
//
// MagicDec notes, section 3.2: verifying gamma draft tokens loads the same KV
// cache as decoding one token, so at long context the verify pass costs about
// one decode step -- the whole point is to read every KV byte once.  This
// kernel therefore processes, for each (sequence, KV head), all G query heads
// of the group and all T = gamma+1 verify rows against each K/V tile while the
// tile sits in shared memory.  The draft pass (quick-read summary and section
// 4.1, Eq. 3: the target itself drafting over a compressed cache of budget K)
// is the same kernel with T = 1 over the compacted cache.
//
// Structure (one CTA = 4 consumer warps + 1 producer warp, 2 CTAs per SM):
//   * work unit = (sequence, KV head, row group, chunk of C keys); a
//     persistent grid pulls units from an atomic counter, so ragged lengths
//     balance themselves and the producer keeps prefetching across units;
//   * the producer streams 64-key K and V tiles with the Tensor Memory
//     Accelerator (128-byte swizzled boxes) into a 3-stage mbarrier ring;
//   * each consumer warp owns 16 keys of every tile and computes
//     S^T = K Q^T with mma.m16n8k16 (keys on the M side, so G*T rows pad only
//     to a multiple of 8), an online softmax in the exp2 domain, and
//     O^T += V^T P^T where P is split into bf16 hi + lo parts (two mmas) so
//     the probabilities keep ~16 significant bits -- or, with three or more
//     n8 row tiles (more than 16 query rows a KV head, as verify at G = 4 and
//     gamma >= 4), one mma in float16: there the mma work per tile is what
//     holds the kernel below the HBM stream (measured at batch 128 x 32k,
//     T = 5: 2.61 ms, 2.39 ms with the QK^T mmas left out, 2.42 ms with the
//     P V ones left out), and P in float16 (11 significant bits for values in
//     [2^-14, 1]) with V converted from bf16 (exact within the float16 range)
//     halves the P V work: 2.51 ms, output rel-L2 1.5e-4 against float64;
//   * at the end of a unit the 4 warps merge in shared memory; a unit that
//     covers the whole sequence writes the final output, otherwise it writes
//     a partial (O, lse) and the CTA that completes the last chunk of that
//     sequence merges all partials (atomic ticket, no waiting).
#include <algorithm>

#include "common.cuh"

namespace mgd {
namespace {

constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBoxBytes = 64 * 128;  // 64 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct TileMeta {
  int unit;
  int tile;
  int ntiles;
  int L;
};

struct KParams {
  int T, Hq, Hkv, G, rows, RG, C, nchunk, kv_cap;
  unsigned total_units;
  float sl2;  // sm_scale * log2(e)
  size_t off_tickets, off_part_o, off_part_l;
};

template <int D, int NT>
struct Layout {
  static constexpr int kBoxes = D / 64;
  static constexpr int kKVBytes = 2 * kBoxes * kBoxBytes;  // K boxes then V boxes
  // With one row tile (at most 8 query rows: the draft pass) the producer also copies a
  // unit's query rows, unpadded, behind the K/V boxes of the stage holding its first tile.
  static constexpr int kQSlotBytes = (NT == 1) ? 8 * D * 2 : 0;
  static constexpr int kStageBytes = kKVBytes + kQSlotBytes;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
  static constexpr int kOStride = 68;                          // epilogue row stride (64 cols + 4)
  static constexpr int kQStride = D + 8;                       // query row stride in bf16 (16 B pad)
  // One buffer serves two phases of a unit: the bf16 query rows while its tiles
  // are processed, then the float32 merge of the 4 warps in its epilogue.
  static constexpr int kEpiBytes = (32 * kOStride * 4 > 32 * kQStride * 2) ? 32 * kOStride * 4 : 32 * kQStride * 2;
  static constexpr int off_epi = kStages * kStageBytes;
  static constexpr int off_m = off_epi + kEpiBytes;  // float [4][32]
  static constexpr int off_l = off_m + 4 * 32 * 4;           // float [4][32]
  static constexpr int off_rowM = off_l + 4 * 32 * 4;        // float [32]
  static constexpr int off_rowL = off_rowM + 32 * 4;         // float [32]
  static constexpr int off_meta = off_rowL + 32 * 4;         // TileMeta [kStages]
  static constexpr int off_bar = off_meta + kStages * 16;    // uint64 full[kStages], empty[kStages]
  static constexpr int off_flag = off_bar + 2 * kStages * 8;
  static constexpr int bytes = off_flag + 16;
  static constexpr int alloc = bytes + 1024;  // slack to align the base to 1024
};

template <int D, int NT, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ kv_len,
                   float *__restrict__ out_f32, __nv_bfloat16 *__restrict__ out_bf16, float *__restrict__ lse_out,
                   unsigned char *__restrict__ ws, KParams p) {
  pdl_launch_dependents();
  using Lay = Layout<D, NT>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *sm_O = reinterpret_cast<float *>(smem + Lay::off_epi);
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + Lay::off_epi);
  float *sm_m = reinterpret_cast<float *>(smem + Lay::off_m);
  float *sm_l = reinterpret_cast<float *>(smem + Lay::off_l);
  float *sm_rowM = reinterpret_cast<float *>(smem + Lay::off_rowM);
  float *sm_rowL = reinterpret_cast<float *>(smem + Lay::off_rowL);
  TileMeta *meta = reinterpret_cast<TileMeta *>(smem + Lay::off_meta);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::off_bar);
  uint64_t *empty = full + kStages;
  int *sm_flag = reinterpret_cast<int *>(smem + Lay::off_flag);

  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  unsigned *tickets = reinterpret_cast<unsigned *>(ws + p.off_tickets);
  float *part_o = reinterpret_cast<float *>(ws + p.off_part_o);
  float *part_l = reinterpret_cast<float *>(ws + p.off_part_l);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    // While the previous kernel in the stream finishes, warm L2 with the first two K and V
    // tiles of this CTA's first unit (its own index; rows past the sequence or the capacity
    // cost nothing but the fetch; more tiles compete with the finishing kernel: measured).
    // Only prefetches: nothing is read before the wait below.
    const int u = static_cast<int>(blockIdx.x);
    const int bh = (u / p.nchunk) / p.RG;
    const int row0 = (u % p.nchunk) * p.C;
    for (int t = 0; t < 2; ++t)
      for (int h = 0; h < Lay::kBoxes; ++h) {
        tma_prefetch_l2_4d(&kmap, h * 64, row0 + t * kTileKeys, bh % p.Hkv, bh / p.Hkv);
        tma_prefetch_l2_4d(&vmap, h * 64, row0 + t * kTileKeys, bh % p.Hkv, bh / p.Hkv);
      }
  }
  __syncthreads();
  pdl_wait();  // set-up above changes no global memory; everything below comes after the previous kernel

  // ====================================================================== producer
  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool first = true;
    unsigned claims = 0;  // successful claims from the counter
    while (ok) {
      // every CTA's first unit is its own index (no counter round trip before the first
      // load); later units come from the counter
      const unsigned u = first ? blockIdx.x : gridDim.x + atomicAdd(&hdr->next_unit, 1u);
      if (u >= p.total_units) break;
      claims += first ? 0u : 1u;
      first = false;
      const int pair = static_cast<int>(u) / p.nchunk;
      const int chunk = static_cast<int>(u) % p.nchunk;
      const int bh = pair / p.RG;
      const int hkv = bh % p.Hkv;
      const int b = bh / p.Hkv;
      const int L = kv_len[b];
      if (L < p.T || L > p.kv_cap) {
        if (chunk == 0) raise_error_sr(hdr, 0x1u);
        continue;
      }
      const int start = chunk * p.C;
      if (start >= L) continue;
      const int end = min(start + p.C, L);
      const int ntiles = (end - start + kTileKeys - 1) / kTileKeys;
      if (NT > 1) {  // warm L2 with this unit's query rows; the consumers load them at its first tile
        const int rg = pair % p.RG;
        const int r_hi = min(p.rows, rg * 32 + 32);
        for (int qg = rg * 32; qg < r_hi; ++qg) {
          const __nv_bfloat16 *qr = q + ((static_cast<size_t>(b) * p.T + qg / p.G) * p.Hq + hkv * p.G + qg % p.G) * D;
          for (int off = 0; off < D * 2; off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(qr) + off));
        }
      }
      for (int t = 0; t < ntiles; ++t) {
        if (!mbar_wait(&empty[stage], phase ^ 1u)) {
          raise_error_sr(hdr, 0x8u);
          ok = false;
          break;
        }
        meta[stage] = TileMeta{static_cast<int>(u), t, ntiles, L};
        const uint32_t qbytes = (Lay::kQSlotBytes > 0 && t == 0) ? static_cast<uint32_t>(p.rows * D * 2) : 0u;
        mbar_arrive_expect_tx(&full[stage], Lay::kKVBytes + qbytes);
        unsigned char *st = smem + stage * Lay::kStageBytes;
        if (qbytes) {  // rows ordered (t, g) like the row index qg = t * G + g
          for (int r = 0; r < p.rows; ++r)
            bulk_load(st + Lay::kKVBytes + r * D * 2,
                      q + ((static_cast<size_t>(b) * p.T + r / p.G) * p.Hq + hkv * p.G + r % p.G) * D, D * 2,
                      &full[stage]);
        }
        const int row = start + t * kTileKeys;
#pragma unroll
        for (int h = 0; h < Lay::kBoxes; ++h) tma_load_4d(st + h * kBoxBytes, &kmap, &full[stage], h * 64, row, hkv, b);
#pragma unroll
        for (int h = 0; h < Lay::kBoxes; ++h)
          tma_load_4d(st + (Lay::kBoxes + h) * kBoxBytes, &vmap, &full[stage], h * 64, row, hkv, b);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (ok && mbar_wait(&empty[stage], phase ^ 1u)) {
      meta[stage].unit = -1;
      mbar_arrive(&full[stage]);
    } else {
      raise_error_sr(hdr, 0x8u);
      // drain: wait (bounded) for every load still in flight before leaving
      for (int s = 0; s < kStages; ++s) mbar_wait(&full[s], phase);
    }
    // This CTA's claims are over: it checks in (its consumers need not: they claim nothing,
    // and their only error bits, timeouts, land in one of the two words either way).
    // From a ready header the counter hands out exactly the units past the first wave.
    call_check_in(hdr, gridDim.x, blockIdx.x, claims, p.total_units - gridDim.x);
    return;
  }

  // ====================================================================== consumers
  const int gid = lane >> 2;
  const int tig = lane & 3;
  constexpr int MT = D / 16;  // m16 tiles over D (PV) == k16 steps over D (QK)
  constexpr bool kF16PV = NT >= 3;  // P V in one float16 mma (see the header)

  float acc[MT][NT][4];
  float m_run[NT][2], l_run[NT][2];
  int lim[NT][2];

  int stage = 0;
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait(&full[stage], phase)) {
      raise_error_sr(hdr, 0x8u);
      break;
    }
    const TileMeta md = meta[stage];
    if (md.unit < 0) break;
    const int pair = md.unit / p.nchunk;
    const int chunk = md.unit % p.nchunk;
    const int rg = pair % p.RG;
    const int bh = pair / p.RG;
    const int hkv = bh % p.Hkv;
    const int b = bh / p.Hkv;
    const int L = md.L;
    const int start = chunk * p.C;

    if (md.tile == 0) {
      // ---- new unit: stage its query rows (zero padded) in shared memory for the
      //      B operand of S^T = K Q^T, and reset the running state
      if constexpr (NT == 1) {
        // rows 0..15 (the ldmatrix.x4 of the QK loop reads two n8 tiles) from the
        // stage's query slot
        const unsigned char *qs = smem + stage * Lay::kStageBytes + Lay::kKVBytes;
        for (int i = threadIdx.x; i < 16 * (D / 8); i += kConsumerWarps * 32) {
          const int r = i / (D / 8), c = i % (D / 8);
          uint4 val = make_uint4(0u, 0u, 0u, 0u);
          if (r < p.rows) val = *reinterpret_cast<const uint4 *>(qs + r * D * 2 + 16 * c);
          *reinterpret_cast<uint4 *>(sQ + r * Lay::kQStride + 8 * c) = val;
        }
      } else {
        // 32 rows from global memory: every load of this thread first, then the stores
        constexpr int kPer = 32 * (D / 8) / (kConsumerWarps * 32);
        uint4 val[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = threadIdx.x + k * kConsumerWarps * 32;
          const int r = i / (D / 8), c = i % (D / 8);
          const int qg = rg * 32 + r;
          val[k] = make_uint4(0u, 0u, 0u, 0u);
          if (qg < p.rows) {
            const int t = qg / p.G, g = qg % p.G;
            val[k] = *reinterpret_cast<const uint4 *>(
                q + ((static_cast<size_t>(b) * p.T + t) * p.Hq + hkv * p.G + g) * D + 8 * c);
          }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = threadIdx.x + k * kConsumerWarps * 32;
          *reinterpret_cast<uint4 *>(sQ + (i / (D / 8)) * Lay::kQStride + 8 * (i % (D / 8))) = val[k];
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int qg = rg * 32 + 8 * j + 2 * tig + e;
          lim[j][e] = (qg < p.rows) ? (L - p.T + qg / p.G) : (L - 1);
          m_run[j][e] = -INFINITY;
          l_run[j][e] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[mt][j][c] = 0.f;
      }
      named_bar(1, kConsumerWarps * 32);
    }

    unsigned char *st = smem + stage * Lay::kStageBytes;
    const int key0 = start + md.tile * kTileKeys + warp * 16;
    bool released = false;  // this warp has handed the stage back to the producer
    if (key0 < L) {
      // ---- S^T[16 keys][8*NT rows] = K Q^T
      float s[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[j][c] = 0.f;
      const uint32_t kbase = smem_addr(st);
      const int kr = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      // B fragments of two n8 row tiles per ldmatrix.x4: rows 16*jp + (lane&7) + 8*(lane>>4)
      const uint32_t qaddr = smem_addr(sQ) + 2u * (((lane & 7) + 8 * (lane >> 4)) * Lay::kQStride + 8 * ((lane >> 3) & 1));
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        const int d = 16 * kk + 8 * (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (d >> 6) * kBoxBytes + swz128(kr, (d & 63) >> 3), a0, a1, a2, a3);
#pragma unroll
        for (int jp = 0; jp < (NT + 1) / 2; ++jp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(qaddr + 2u * (16 * jp * Lay::kQStride + 16 * kk), b0, b1, b2, b3);
          mma_bf16_16816(s[2 * jp], a0, a1, a2, a3, b0, b1);
          if (2 * jp + 1 < NT) mma_bf16_16816(s[2 * jp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- rows past the sequence end hold stale bytes: zero this warp's V rows there
      if (key0 + 16 > L) {
        const int r0 = L - key0;  // first invalid local row (1..15)
        const int nchunks = (16 - r0) * 8 * Lay::kBoxes;
        for (int i = lane; i < nchunks; i += 32) {
          const int h = i / ((16 - r0) * 8);
          const int rem = i % ((16 - r0) * 8);
          const int r = warp * 16 + r0 + rem / 8;
          const int c = rem % 8;
          *reinterpret_cast<uint4 *>(st + (Lay::kBoxes + h) * kBoxBytes + swz128(r, c)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // ---- this warp's V^T fragments into registers, then the stage goes back to the
      //      producer: the softmax and O^T += V^T P^T below no longer hold it, so the
      //      ring keeps more tiles in flight
      uint32_t va[MT][4];
      {
        const uint32_t vbase = smem_addr(st + Lay::kBoxes * kBoxBytes);
        const int vr = warp * 16 + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int d = 16 * mt + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(vbase + (d >> 6) * kBoxBytes + swz128(vr, (d & 63) >> 3), va[mt][0], va[mt][1], va[mt][2],
                    va[mt][3]);
          if constexpr (kF16PV) {
#pragma unroll
            for (int c = 0; c < 4; ++c) va[mt][c] = bf16x2_to_f16x2(va[mt][c]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      released = true;
      // ---- scale, mask, online softmax (exp2 domain)
      const bool need_mask = key0 + 15 > L - p.T;
      const int k_lo = key0 + gid, k_hi = key0 + gid + 8;
      uint32_t phi[NT][2], plo[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float alpha[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v0 = s[j][e] * p.sl2;
          float v1 = s[j][2 + e] * p.sl2;
          if (need_mask) {
            if (k_lo > lim[j][e]) v0 = -INFINITY;
            if (k_hi > lim[j][e]) v1 = -INFINITY;
          }
          const float mx = warp_max_xor(fmaxf(v0, v1), 4, 16);
          const float mnew = fmaxf(m_run[j][e], mx);
          const float muse = (mnew == -INFINITY) ? 0.f : mnew;
          alpha[e] = ex2(m_run[j][e] - muse);
          const float p0 = ex2(v0 - muse);
          const float p1 = ex2(v1 - muse);
          l_run[j][e] = l_run[j][e] * alpha[e] + p0 + p1;
          m_run[j][e] = mnew;
          s[j][e] = p0;
          s[j][2 + e] = p1;
        }
        const float2 a2 = make_float2(alpha[0], alpha[1]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {  // paired (f32x2) multiplies: columns 2 tig, 2 tig + 1
          const float2 x = __fmul2_rn(make_float2(acc[mt][j][0], acc[mt][j][1]), a2);
          const float2 y = __fmul2_rn(make_float2(acc[mt][j][2], acc[mt][j][3]), a2);
          acc[mt][j][0] = x.x;
          acc[mt][j][1] = x.y;
          acc[mt][j][2] = y.x;
          acc[mt][j][3] = y.y;
        }
        if constexpr (kF16PV) {
          phi[j][0] = movmatrix_t(pack_f16(s[j][0], s[j][1]));  // keys gid,   rows 2tig, 2tig+1
          phi[j][1] = movmatrix_t(pack_f16(s[j][2], s[j][3]));  // keys gid+8, rows 2tig, 2tig+1
        } else {
          uint32_t h0, l0, h1, l1;
          split_bf16(s[j][0], s[j][1], h0, l0);  // keys gid,   rows 2tig, 2tig+1
          split_bf16(s[j][2], s[j][3], h1, l1);  // keys gid+8, rows 2tig, 2tig+1
          phi[j][0] = movmatrix_t(h0);
          phi[j][1] = movmatrix_t(h1);
          plo[j][0] = movmatrix_t(l0);
          plo[j][1] = movmatrix_t(l1);
        }
      }
      // ---- O^T[D][rows] += V^T P^T
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if constexpr (kF16PV) {
            mma_f16_16816(acc[mt][j], va[mt][0], va[mt][1], va[mt][2], va[mt][3], phi[j][0], phi[j][1]);
          } else {
            mma_bf16_16816(acc[mt][j], va[mt][0], va[mt][1], va[mt][2], va[mt][3], phi[j][0], phi[j][1]);
            mma_bf16_16816(acc[mt][j], va[mt][0], va[mt][1], va[mt][2], va[mt][3], plo[j][0], plo[j][1]);
          }
        }
      }
    }
    if (!released) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (md.tile != md.ntiles - 1) continue;

    // ================================================================ unit epilogue
    const int rows_valid = min(32, p.rows - rg * 32);
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) l_run[j][e] = warp_sum_xor(l_run[j][e], 4, 16);
    if (gid == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sm_m[warp * 32 + 8 * j + 2 * tig + e] = m_run[j][e];
          sm_l[warp * 32 + 8 * j + 2 * tig + e] = l_run[j][e];
        }
    }
    named_bar(1, kConsumerWarps * 32);
    if (threadIdx.x < 32) {
      const int r = threadIdx.x;
      float M = -INFINITY;
      for (int w = 0; w < kConsumerWarps; ++w)
        if (r < 8 * NT) M = fmaxf(M, sm_m[w * 32 + r]);
      const float Mu = (M == -INFINITY) ? 0.f : M;
      float Lt = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w)
        if (r < 8 * NT) Lt += sm_l[w * 32 + r] * exp2f(sm_m[w * 32 + r] - Mu);
      sm_rowM[r] = Mu;
      sm_rowL[r] = Lt;
    }
    named_bar(1, kConsumerWarps * 32);
    float f[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) f[j][e] = exp2f(m_run[j][e] - sm_rowM[8 * j + 2 * tig + e]);

    const int nch_b = (L + p.C - 1) / p.C;
    const bool single = (nch_b == 1);
    const size_t part_base = (static_cast<size_t>(pair) * p.nchunk + chunk) * 32;
    // The 4 warps' scaled accumulators meet in kSlices slices of 8*NT rows (as many as the
    // 32-row buffer holds): the warps of round 0 store their slice, later rounds add into
    // it in turn, and the write-out sums the slices -- no shared-memory atomics.
    constexpr int kSlices = (NT == 1) ? 4 : (NT == 2) ? 2 : 1;
    constexpr int kRounds = kConsumerWarps / kSlices;
    float *my_slice = sm_O + (warp % kSlices) * (8 * NT) * Lay::kOStride;
#pragma unroll
    for (int dh = 0; dh < D / 64; ++dh) {
#pragma unroll
      for (int rd = 0; rd < kRounds; ++rd) {
        if (warp / kSlices == rd) {
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const int mt = dh * 4 + mm;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float *o0 = my_slice + (8 * j + 2 * tig + e) * Lay::kOStride + 16 * mm + gid;
                const float v0 = acc[mt][j][e] * f[j][e], v1 = acc[mt][j][2 + e] * f[j][e];
                if (rd == 0) {
                  o0[0] = v0;
                  o0[8] = v1;
                } else {
                  o0[0] += v0;
                  o0[8] += v1;
                }
              }
          }
        }
        named_bar(1, kConsumerWarps * 32);
      }
      for (int i = threadIdx.x; i < rows_valid * 16; i += kConsumerWarps * 32) {
        const int r = i >> 4, dq = i & 15;
        const float Lt = sm_rowL[r];
        const float inv = (Lt > 0.f) ? 1.f / Lt : 0.f;
        float4 o = *reinterpret_cast<const float4 *>(&sm_O[r * Lay::kOStride + 4 * dq]);
#pragma unroll
        for (int sl = 1; sl < kSlices; ++sl) {
          const float4 x = *reinterpret_cast<const float4 *>(&sm_O[(sl * 8 * NT + r) * Lay::kOStride + 4 * dq]);
          o.x += x.x;
          o.y += x.y;
          o.z += x.z;
          o.w += x.w;
        }
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        const int d = dh * 64 + 4 * dq;
        const int qg = rg * 32 + r;
        if (single) {
          const int t = qg / p.G, g = qg % p.G;
          const size_t orow = (static_cast<size_t>(b) * p.T + t) * p.Hq + hkv * p.G + g;
          if (out_bf16) {
            uint2 pk;
            pk.x = pack_bf16(o.x, o.y);
            pk.y = pack_bf16(o.z, o.w);
            *reinterpret_cast<uint2 *>(out_bf16 + orow * D + d) = pk;
          } else {
            *reinterpret_cast<float4 *>(out_f32 + orow * D + d) = o;
          }
          if (lse_out && dh == 0 && dq == 0)
            lse_out[orow] = (Lt > 0.f) ? (sm_rowM[r] + log2f(Lt)) * kLn2 : -INFINITY;
        } else {
          *reinterpret_cast<float4 *>(part_o + (part_base + r) * D + d) = o;
          if (dh == 0 && dq == 0) part_l[part_base + r] = (Lt > 0.f) ? (sm_rowM[r] + log2f(Lt)) * kLn2 : -INFINITY;
        }
      }
      named_bar(1, kConsumerWarps * 32);
    }
    if (single) continue;

    // ---- the CTA that finishes the last chunk of this pair merges all partials
    __threadfence();
    named_bar(1, kConsumerWarps * 32);
    if (threadIdx.x == 0) {
      const unsigned old = atomicAdd(&tickets[pair], 1u);
      const bool last = (old == static_cast<unsigned>(nch_b - 1));
      if (last) tickets[pair] = 0u;  // every chunk of the pair has arrived: ready for the next call
      *sm_flag = last ? 1 : 0;
    }
    named_bar(1, kConsumerWarps * 32);
    if (*sm_flag) {
      __threadfence();
      const size_t pb0 = static_cast<size_t>(pair) * p.nchunk * 32;
      // all chunk lse values at once (independent loads), then per-row weights
      float *sm_w = sm_O;  // [nch_b][32]; the epilogue buffer is free again
      for (int i = threadIdx.x; i < nch_b * 32; i += kConsumerWarps * 32)
        sm_w[i] = ((i & 31) < rows_valid) ? __ldcg(part_l + pb0 + i) : -INFINITY;
      named_bar(1, kConsumerWarps * 32);
      if (threadIdx.x < rows_valid) {
        const int r = threadIdx.x;
        float M = -INFINITY;
        for (int c = 0; c < nch_b; ++c) M = fmaxf(M, sm_w[c * 32 + r]);
        float W = 0.f;
        for (int c = 0; c < nch_b; ++c) {
          const float w = expf(sm_w[c * 32 + r] - M);
          sm_w[c * 32 + r] = w;
          W += w;
        }
        for (int c = 0; c < nch_b; ++c) sm_w[c * 32 + r] /= W;
        sm_rowM[r] = M;
        sm_rowL[r] = W;
      }
      named_bar(1, kConsumerWarps * 32);
      for (int i = threadIdx.x; i < rows_valid * (D / 4); i += kConsumerWarps * 32) {
        const int r = i / (D / 4), dq = i % (D / 4);
        const float M = sm_rowM[r];
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < nch_b; c0 += 8) {  // 8 independent loads in flight per thread
          float4 x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            x[u] = (c0 + u < nch_b)
                       ? __ldcg(reinterpret_cast<const float4 *>(part_o + (pb0 + (c0 + u) * 32 + r) * D + 4 * dq))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float w = (c0 + u < nch_b) ? sm_w[(c0 + u) * 32 + r] : 0.f;
            o.x += w * x[u].x;
            o.y += w * x[u].y;
            o.z += w * x[u].z;
            o.w += w * x[u].w;
          }
        }
        const int qg = rg * 32 + r;
        const int t = qg / p.G, g = qg % p.G;
        const size_t orow = (static_cast<size_t>(b) * p.T + t) * p.Hq + hkv * p.G + g;
        if (out_bf16) {
          uint2 pk;
          pk.x = pack_bf16(o.x, o.y);
          pk.y = pack_bf16(o.z, o.w);
          *reinterpret_cast<uint2 *>(out_bf16 + orow * D + 4 * dq) = pk;
        } else {
          *reinterpret_cast<float4 *>(out_f32 + orow * D + 4 * dq) = o;
        }
        if (lse_out && dq == 0) lse_out[orow] = M + logf(sm_rowL[r]);
      }
      named_bar(1, kConsumerWarps * 32);
    }
  }
}

template <int D, int NT>
cudaError_t launch_one(const AttnPlan &pl, const AttnArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap) {
  constexpr int MINB = (NT <= 3) ? 2 : 1;
  auto kern = attn_tc_kernel<D, NT, MINB>;
  const int smem = Layout<D, NT>::alloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  KParams kp;
  kp.T = pl.T;
  kp.Hq = pl.Hq;
  kp.Hkv = pl.Hkv;
  kp.G = pl.G;
  kp.rows = pl.rows;
  kp.RG = pl.RG;
  kp.C = pl.C;
  kp.nchunk = pl.nchunk;
  kp.kv_cap = pl.kv_cap;
  kp.total_units = static_cast<unsigned>(pl.pairs) * static_cast<unsigned>(pl.nchunk);
  kp.sl2 = a.sm_scale * kLog2e;
  kp.off_tickets = pl.off_tickets;
  kp.off_part_o = pl.off_part_o;
  kp.off_part_l = pl.off_part_l;
  // one persistent CTA per resident slot (MINB per SM unless shared memory allows fewer)
  static const int resident = [&] {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads, smem) != cudaSuccess) nb = MINB;
    return std::max(1, std::min(nb, MINB));
  }();
  int grid = pl.grid / MINB * resident;
  if (static_cast<unsigned>(grid) > kp.total_units) grid = static_cast<int>(kp.total_units);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, a.stream, kmap, vmap,
                    static_cast<const __nv_bfloat16 *>(a.q), a.kv_len,
                    a.out_bf16 ? nullptr : static_cast<float *>(a.out),
                    a.out_bf16 ? static_cast<__nv_bfloat16 *>(a.out) : nullptr, a.lse,
                    static_cast<unsigned char *>(a.ws), kp);
}

}  // namespace

int attn_tc_min_blocks(int NT) { return NT <= 3 ? 2 : 1; }

cudaError_t launch_attention_tc(const AttnPlan &pl, const AttnArgs &a, const CUtensorMap &kmap,
                                const CUtensorMap &vmap) {
  // The header needs no clearing launch: the kernel leaves it ready for the next call
  // (the workspace is zero-filled before its first use).  The merge tickets of split
  // sequences are cleared here, since a call of another shape may have written
  // partial results where this call keeps them.
  if (pl.nchunk > 1) {
    cudaError_t e = cudaMemsetAsync(static_cast<unsigned char *>(a.ws) + pl.off_tickets, 0,
                                    pl.off_part_o - pl.off_tickets, a.stream);
    if (e != cudaSuccess) return e;
  }
  if (pl.D == 128) {
    switch (pl.NT) {
      case 1: return launch_one<128, 1>(pl, a, kmap, vmap);
      case 2: return launch_one<128, 2>(pl, a, kmap, vmap);
      case 3: return launch_one<128, 3>(pl, a, kmap, vmap);
      default: return launch_one<128, 4>(pl, a, kmap, vmap);
    }
  } else {
    switch (pl.NT) {
      case 1: return launch_one<64, 1>(pl, a, kmap, vmap);
      case 2: return launch_one<64, 2>(pl, a, kmap, vmap);
      case 3: return launch_one<64, 3>(pl, a, kmap, vmap);
      default: return launch_one<64, 4>(pl, a, kmap, vmap);
    }
  }
}

AttnPlan plan_attention(int B, int T, int Hq, int Hkv, int D, int kv_cap, int sm_count) {
  AttnPlan p{};
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.kv_cap = kv_cap;
  p.G = Hq / Hkv;
  p.rows = p.G * T;
  p.RG = (p.rows + 31) / 32;
  p.rows_pg = p.RG == 1 ? p.rows : 32;
  p.NT = (p.rows_pg + 7) / 8;
  p.pairs = B * Hkv * p.RG;
  const int slots = attn_tc_min_blocks(p.NT) * sm_count;
  // Largest power-of-two chunk (<= 16384 keys) that still leaves >= 3 units per
  // persistent CTA: every unit pays a query load, an epilogue and (when the
  // sequence is split) a partial write and merge, so fewer, longer units win
  // until the last wave's imbalance dominates.  At most 64 chunks per pair
  // (the merge keeps one weight per chunk in shared memory).
  // When every pair fits in one wave of CTA slots, whole sequences (up to
  // 16384 keys) win: splitting buys no balance and costs partial writes and
  // merges (measured at batch 32: draft 32.5 -> 23.0 us, verify over 8k and
  // 16k keys 0.215 -> 0.172 ms and 0.373 -> 0.320 ms).
  int C = 16384;
  const int cmin = std::max(256, ((kv_cap + 63) / 64 + 63) / 64 * 64);
  if (p.pairs > slots)
    while (C > cmin && static_cast<long long>(p.pairs) * ((kv_cap + C - 1) / C) < 3LL * slots) C /= 2;
  if (C < cmin) C = cmin;
  p.C = C;
  p.nchunk = (kv_cap + C - 1) / C;
  p.grid = slots;
  size_t off = kAlign;  // header
  p.off_tickets = off;
  off = align_up(off + sizeof(unsigned) * static_cast<size_t>(p.pairs));
  p.off_part_o = off;
  const size_t nparts = (p.nchunk > 1) ? static_cast<size_t>(p.pairs) * p.nchunk * 32 : 0;
  off = align_up(off + nparts * D * sizeof(float));
  p.off_part_l = off;
  off = align_up(off + nparts * sizeof(float));
  p.ws_bytes = off;
  return p;
}

}  // namespace mgd
