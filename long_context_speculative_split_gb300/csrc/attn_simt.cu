// CUDA-core attention for float32 inputs: the float32 instantiation
// of the verify / draft pass.  Same definition as the tensor-core kernel
// (MagicDec notes, section 3.2: verify = decode attention over gamma+1 rows;
// causal among the appended rows), float32 arithmetic throughout.  One CTA
// per (sequence, KV head); each warp walks a strided subset of the keys with
// an online softmax and the 4 warps merge in shared memory.  It is the
// correctness path for float32 inputs, not the timed bf16 path.
#include "common.cuh"

namespace mgd {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerPass = 8;

template <typename Tin, int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                     const int32_t *__restrict__ kv_len, int T, int Hq, int Hkv, int G, int kv_cap,
                     int64_t bstride, int64_t hstride, float sl2, float *__restrict__ out_f32,
                     __nv_bfloat16 *__restrict__ out_bf16, float *__restrict__ lse_out, WsHeader *hdr) {
  constexpr int E = D / 32;
  __shared__ float sm_m[kWarps][kRowsPerPass];
  __shared__ float sm_l[kWarps][kRowsPerPass];
  __shared__ float sm_o[kWarps][kRowsPerPass][D];

  const int b = blockIdx.x / Hkv;
  const int hkv = blockIdx.x % Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = kv_len[b];
  if (L < T || L > kv_cap) {
    if (threadIdx.x == 0 && hkv == 0) raise_error(hdr, 0x1u);
    return;
  }
  const int rows = G * T;
  const Tin *kb = k + b * bstride + hkv * hstride;
  const Tin *vb = v + b * bstride + hkv * hstride;

  for (int rb = 0; rb < rows; rb += kRowsPerPass) {
    float qv[kRowsPerPass][E], o[kRowsPerPass][E], m[kRowsPerPass], l[kRowsPerPass];
    int lim[kRowsPerPass];
#pragma unroll
    for (int i = 0; i < kRowsPerPass; ++i) {
      const int r = rb + i;
      m[i] = -INFINITY;
      l[i] = 0.f;
      lim[i] = -1;
      if (r < rows) {
        const int t = r / G, g = r % G;
        lim[i] = L - T + t;
        const Tin *qr = q + ((static_cast<size_t>(b) * T + t) * Hq + hkv * G + g) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) qv[i][e] = to_f32(qr[lane + 32 * e]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) qv[i][e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) o[i][e] = 0.f;
    }
    for (int j = warp; j < L; j += kWarps) {
      float kv[E], vv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kv[e] = to_f32(kb[static_cast<size_t>(j) * D + lane + 32 * e]);
        vv[e] = to_f32(vb[static_cast<size_t>(j) * D + lane + 32 * e]);
      }
#pragma unroll
      for (int i = 0; i < kRowsPerPass; ++i) {
        if (j > lim[i]) continue;  // warp-uniform
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qv[i][e], kv[e], dot);
        dot = warp_sum_xor(dot, 1, 16);
        const float s = dot * sl2;
        const float mn = fmaxf(m[i], s);
        const float alpha = exp2f(m[i] - mn);
        const float pj = exp2f(s - mn);
        l[i] = l[i] * alpha + pj;
#pragma unroll
        for (int e = 0; e < E; ++e) o[i][e] = o[i][e] * alpha + pj * vv[e];
        m[i] = mn;
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerPass; ++i) {
      if (lane == 0) {
        sm_m[warp][i] = m[i];
        sm_l[warp][i] = l[i];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) sm_o[warp][i][lane + 32 * e] = o[i][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kRowsPerPass * D; idx += kWarps * 32) {
      const int i = idx / D, d = idx % D;
      const int r = rb + i;
      if (r >= rows) continue;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][i]);
      float Lt = 0.f, acc = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        const float f = (sm_m[w][i] == -INFINITY) ? 0.f : exp2f(sm_m[w][i] - M);
        Lt += sm_l[w][i] * f;
        acc += sm_o[w][i][d] * f;
      }
      const int t = r / G, g = r % G;
      const size_t orow = (static_cast<size_t>(b) * T + t) * Hq + hkv * G + g;
      const float val = acc / Lt;
      if (out_bf16)
        out_bf16[orow * D + d] = __float2bfloat16_rn(val);
      else
        out_f32[orow * D + d] = val;
      if (lse_out && d == 0) lse_out[orow] = (M + log2f(Lt)) * 0.6931471805599453f;
    }
    __syncthreads();
  }
}

}  // namespace

size_t simt_attention_ws_bytes() { return kAlign; }

cudaError_t launch_attention_simt(const AttnPlan &p, const AttnArgs &a) {
  cudaError_t e = cudaMemsetAsync(a.ws, 0, kAlign, a.stream);
  if (e != cudaSuccess) return e;
  const float sl2 = a.sm_scale * 1.4426950408889634f;
  float *of = a.out_bf16 ? nullptr : static_cast<float *>(a.out);
  __nv_bfloat16 *ob = a.out_bf16 ? static_cast<__nv_bfloat16 *>(a.out) : nullptr;
  WsHeader *hdr = static_cast<WsHeader *>(a.ws);
  const int grid = p.B * p.Hkv;
#define MGD_SIMT(TY, DD)                                                                                     \
  attn_simt_kernel<TY, DD><<<grid, kWarps * 32, 0, a.stream>>>(                                              \
      static_cast<const TY *>(a.q), static_cast<const TY *>(a.k), static_cast<const TY *>(a.v), a.kv_len, p.T, \
      p.Hq, p.Hkv, p.G, p.kv_cap, a.kv_batch_stride, a.kv_head_stride, sl2, of, ob, a.lse, hdr)
  if (p.D == 128)
    MGD_SIMT(float, 128);
  else
    MGD_SIMT(float, 64);
#undef MGD_SIMT
  return cudaGetLastError();
}

}  // namespace mgd
