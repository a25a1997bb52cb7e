// kda_decode.cu -- one decode step of the KDA recurrence for a batch of rows.
//
// "Kimi K3: The Manos, The Mythos, The Legendos" (bullet on FlashKDA): decode
// costs the same at every position because each step only advances a
// fixed-size state by one token.  Per (row, head) the step is
//
//   S' = Diag(alpha) S                 p = S'^T k^       u = beta (v - p)
//   S  = S' + k^ u^T                   o = scale S^T q^ = scale (S'^T q^ + (q^.k^) u)
//
// (delta rule with a per-channel gate, "From KV Cache to Depth Attention",
// Technical Details).  The work is ~7 dk dv flops per 8 dk dv bytes of state
// traffic, so the kernel is bound by HBM: it reads the fp32 state once into
// registers with 16-byte coalesced loads (a warp covers whole 512-byte rows
// for dv = 128), reduces S'^T k^ and S'^T q^ over the key channels in
// registers and through shared memory, and writes the state back once.
#include "kda_internal.cuh"

namespace kda {
namespace {

template <typename TIn, int DK, int DV>
struct DecodeShape {
  static constexpr int QPR = DV / 4;                           // float4 quads per row
  static constexpr int NT = (QPR * DK < 256) ? QPR * DK : 256; // threads
  static constexpr int NRG = NT / QPR;                         // row groups
  static constexpr int RPT = DK / NRG;                         // rows per thread
  static_assert(DK % NRG == 0, "row groups tile the key channels");
};

template <typename TIn, int DK, int DV>
__global__ void __launch_bounds__(DecodeShape<TIn, DK, DV>::NT)
decode_step(kda_decode_args a) {
  using Sh = DecodeShape<TIn, DK, DV>;
  constexpr int QPR = Sh::QPR, NT = Sh::NT, NRG = Sh::NRG, RPT = Sh::RPT;
  __shared__ float qn[DK], kn[DK], al[DK], vv[DV];
  __shared__ float red_p[NRG][DV], red_o[NRG][DV];
  __shared__ float sc[2];  // beta, q^.k^

  const int row = blockIdx.x, h = blockIdx.y, H = a.num_heads;
  const int slot = a.state_slots ? a.state_slots[row] : row;
  if (slot < 0 || slot >= a.num_slots) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % QPR, rg = tid / QPR;
  float* S = a.state + ((size_t)slot * H + h) * DK * DV;

  // stream this thread's rows of the state into registers first
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    s[i] = reinterpret_cast<const float4*>(S + (size_t)(rg + i * NRG) * DV)[cq];

  // token preparation (one warp): q^, k^, alpha, beta, q^.k^
  if (warp == 0) {
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* g = static_cast<const TIn*>(a.g);
    const TIn* v = static_cast<const TIn*>(a.v);
    const int64_t base_k = ((int64_t)row * H + h) * DK;
    const int64_t base_v = ((int64_t)row * H + h) * DV;
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < DK; c += 32) {
      const float xq = ld_in(q, base_k + c), xk = ld_in(k, base_k + c);
      qn[c] = xq;
      kn[c] = xk;
      al[c] = expf(log_alpha_of(ld_in(g, base_k + c)));
      sq += xq * xq;
      sk += xk * xk;
    }
    for (int c = lane; c < DV; c += 32) vv[c] = ld_in(v, base_v + c);
    const float iq = inv_norm_of(warp_sum(sq)), ik = inv_norm_of(warp_sum(sk));
    float qk = 0.f;
    for (int c = lane; c < DK; c += 32) {
      qn[c] *= iq;
      kn[c] *= ik;
      qk += qn[c] * kn[c];
    }
    qk = warp_sum(qk);
    if (lane == 0) {
      sc[0] = beta_of(ld_in(static_cast<const TIn*>(a.b), (int64_t)row * H + h));
      sc[1] = qk;
    }
  }
  __syncthreads();

  // retention and the two reductions over key channels
  float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), po = pp;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * NRG;
    const float a_r = al[r], k_r = kn[r], q_r = qn[r];
    s[i].x *= a_r; s[i].y *= a_r; s[i].z *= a_r; s[i].w *= a_r;
    pp.x += k_r * s[i].x; pp.y += k_r * s[i].y; pp.z += k_r * s[i].z; pp.w += k_r * s[i].w;
    po.x += q_r * s[i].x; po.y += q_r * s[i].y; po.z += q_r * s[i].z; po.w += q_r * s[i].w;
  }
  // row groups that share a warp (dv < 128) combine with shuffles first
  constexpr int RGW = 32 / QPR;  // row groups per warp
#pragma unroll
  for (int off = QPR; off < 32 && RGW > 1; off <<= 1) {
    pp.x += __shfl_xor_sync(0xffffffffu, pp.x, off);
    pp.y += __shfl_xor_sync(0xffffffffu, pp.y, off);
    pp.z += __shfl_xor_sync(0xffffffffu, pp.z, off);
    pp.w += __shfl_xor_sync(0xffffffffu, pp.w, off);
    po.x += __shfl_xor_sync(0xffffffffu, po.x, off);
    po.y += __shfl_xor_sync(0xffffffffu, po.y, off);
    po.z += __shfl_xor_sync(0xffffffffu, po.z, off);
    po.w += __shfl_xor_sync(0xffffffffu, po.w, off);
  }
  constexpr int NW = NT / 32 > 0 ? NT / 32 : 1;
  const bool writer = (RGW > 1) ? (lane < QPR) : true;
  const int slotw = (RGW > 1) ? warp : rg;
  if (writer) {
    *reinterpret_cast<float4*>(&red_p[slotw][4 * cq]) = pp;
    *reinterpret_cast<float4*>(&red_o[slotw][4 * cq]) = po;
  }
  __syncthreads();
  const int nred = (RGW > 1) ? NW : NRG;
  float4 p = make_float4(0.f, 0.f, 0.f, 0.f), oq = p;
  for (int w = 0; w < nred; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(&red_p[w][4 * cq]);
    const float4 y = *reinterpret_cast<const float4*>(&red_o[w][4 * cq]);
    p.x += x.x; p.y += x.y; p.z += x.z; p.w += x.w;
    oq.x += y.x; oq.y += y.y; oq.z += y.z; oq.w += y.w;
  }
  const float beta = sc[0];
  const float4 vq = *reinterpret_cast<const float4*>(&vv[4 * cq]);
  const float4 u = make_float4(beta * (vq.x - p.x), beta * (vq.y - p.y), beta * (vq.z - p.z),
                               beta * (vq.w - p.w));
  // rank-1 write of the delta, state written back once
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * NRG;
    const float k_r = kn[r];
    float4 x = s[i];
    x.x += k_r * u.x; x.y += k_r * u.y; x.z += k_r * u.z; x.w += k_r * u.w;
    reinterpret_cast<float4*>(S + (size_t)r * DV)[cq] = x;
  }
  if (rg == 0) {
    const float qk = sc[1], scl = a.scale;
    TIn* o = static_cast<TIn*>(a.o);
    const int64_t ob = ((int64_t)row * H + h) * DV + 4 * cq;
    st_out(o, ob + 0, scl * (oq.x + qk * u.x));
    st_out(o, ob + 1, scl * (oq.y + qk * u.y));
    st_out(o, ob + 2, scl * (oq.z + qk * u.z));
    st_out(o, ob + 3, scl * (oq.w + qk * u.w));
  }
}

template <typename TIn, int DK, int DV>
cudaError_t launch_t(const kda_decode_args& a, cudaStream_t stream) {
  dim3 grid((unsigned)a.batch, (unsigned)a.num_heads);
  decode_step<TIn, DK, DV><<<grid, DecodeShape<TIn, DK, DV>::NT, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename TIn, int DK>
cudaError_t launch_dv(const kda_decode_args& a, cudaStream_t stream) {
  switch (a.dv) {
    case 16: return launch_t<TIn, DK, 16>(a, stream);
    case 32: return launch_t<TIn, DK, 32>(a, stream);
    case 64: return launch_t<TIn, DK, 64>(a, stream);
    case 128: return launch_t<TIn, DK, 128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t launch_dk(const kda_decode_args& a, cudaStream_t stream) {
  switch (a.dk) {
    case 16: return launch_dv<TIn, 16>(a, stream);
    case 32: return launch_dv<TIn, 32>(a, stream);
    case 64: return launch_dv<TIn, 64>(a, stream);
    case 128: return launch_dv<TIn, 128>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const kda_decode_args& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  return a.in_dtype == KDA_BF16 ? launch_dk<__nv_bfloat16>(a, stream) : launch_dk<float>(a, stream);
}

}  // namespace kda
