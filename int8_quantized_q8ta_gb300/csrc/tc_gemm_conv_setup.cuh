// tc_gemm_conv_setup.cuh -- host set-up shared by the two convolution GEMM
// launchers: tile shape, TMA tensor maps and kernel parameters of one group.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "q8ta_internal.h"
#include "tc_gemm_kernel.cuh"

namespace q8 {

inline int64_t gcd64(int64_t a, int64_t b) {
  while (b != 0) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// a^-1 modulo m for coprime a, m (extended Euclid); 0 when m == 1.
inline int64_t inv_mod(int64_t a, int64_t m) {
  if (m == 1) return 0;
  int64_t t = 0, nt = 1, r = m, nr = a % m;
  while (nr != 0) {
    const int64_t q = r / nr;
    const int64_t t2 = t - q * nt;
    t = nt;
    nt = t2;
    const int64_t r2 = r - q * nr;
    r = nr;
    nr = r2;
  }
  return t < 0 ? t + m : t;
}

// Row taps of transposed-convolution phase ph: kh with kh * dil = ph + pad
// (mod stride), kh < K (the count the kernel's decode derives).
inline int conv_t_phase_taps(int64_t ph, int64_t pad, int64_t stride, int64_t dil, int64_t K) {
  const int64_t g = gcd64(dil, stride), ts = stride / g;
  const int64_t t = (ph + pad) % stride;
  if (t % g != 0) return 0;
  const int64_t k0 = (t / g) * inv_mod(dil / g, ts) % ts;
  return k0 < K ? static_cast<int>((K - k0 + ts - 1) / ts) : 0;
}

struct ConvSetup {
  CUtensorMap ma, mb;
  TcParams p;
  int bn, kd;
  bool pixn;    // output channels on the MMA's M side, bn pixels on N
  bool single;  // every sub-tile fits one exact chunk (the host's bounds)
};

// Ring stages per exact f32 chunk, as the kernel's chunk_stages computes it
// from the same bounds.
inline int host_chunk_stages(int a_bound, int w_bound, int kd) {
  if (a_bound < 1 || a_bound > 255) a_bound = 255;
  if (w_bound > kWorstWBound || w_bound < 0) w_bound = kWorstWBound;
  w_bound = std::max(w_bound, 1);
  const int kb = std::min(kMaxChunkKb, (1 << 24) / (a_bound * w_bound));
  return std::max(1, kb / kd);
}

// Pixels of an exchanged-operand tile (the MMA's N).
constexpr int kPixTile = 256;

// Tile shape: tile_px output pixels (bw columns x bh rows of a stride phase
// for the transposed convolution, of the output for the direct one) x the
// output channels of one block.  More than 64 output channels on images of
// at least one exchanged tile per phase: 128 channels (M) x 256 pixels (N);
// otherwise 128 pixels (M) x bn channels (N).  The direct convolution reads
// its input through boxes with element strides (stride_w, stride_h), whose
// extents bw * stride_w and bh * stride_h must stay within the TMA limit of
// 256.
inline bool conv_setup(const TcConvT& C, ConvSetup& S) {
  const bool direct = C.direct;
  const int64_t Hq = direct ? C.H_out : (C.H_out + C.stride_h - 1) / C.stride_h;
  const int64_t Wq = direct ? C.W_out : (C.W_out + C.stride_w - 1) / C.stride_w;
  const int64_t ew = direct ? C.stride_w : 1, eh = direct ? C.stride_h : 1;
  const bool pixn = C.OC > 64 && Hq * Wq >= kPixTile;
  const int bn = pixn ? kPixTile : pick_bn(C.OC);  // the MMA's N
  const int oc_blk = pixn ? kBM : bn;              // output channels per tile
  const int tile_px = pixn ? kPixTile : kBM;
  int bw = 1;
  while (bw < Wq && bw < tile_px) bw *= 2;
  while (bw > 1 && bw * ew > 256) bw /= 2;
  while (bw < tile_px && (tile_px / bw) * eh > 256) bw *= 2;
  const int bh = tile_px / bw;
  if (bw * ew > 256 || bh * eh > 256) return false;
  const uint64_t icb = static_cast<uint64_t>(C.ICp / kBK);
  // the most taps of any sub-tile
  int max_taps = static_cast<int>(C.Kh * C.Kw);
  if (!direct) {
    int th = 0, tw = 0;
    for (int ph = 0; ph < C.stride_h; ++ph)
      th = std::max(th, conv_t_phase_taps(ph, C.pad_h, C.stride_h, C.dil_h, C.Kh));
    for (int pw = 0; pw < C.stride_w; ++pw)
      tw = std::max(tw, conv_t_phase_taps(pw, C.pad_w, C.stride_w, C.dil_w, C.Kw));
    max_taps = th * tw;
  }
  // Two k-blocks (channel blocks) per TMA box when they split evenly: the
  // 128-wide tiles need bigger boxes to keep enough bytes in flight per SM.
  // The exchanged tiles (48 KB per k-block) keep one k-block per stage: four
  // 48 KB stages measured faster than two 96 KB ones (21.2 us against 22.1
  // us for the 8x256x64x64 transposed convolution's GEMM): the feed is bound
  // by bytes from L2, not by the count of boxes.
  const int kd = (!pixn && icb % 2 == 0) ? 2 : 1;
  {
    // the group's channel blocks of [N][cb_total][H_in][W_in][64] bf16
    const uint64_t dims[5] = {kBK, static_cast<uint64_t>(C.W_in), static_cast<uint64_t>(C.H_in),
                              icb, static_cast<uint64_t>(C.N)};
    const uint64_t row = kBK * 2;
    const uint64_t str[4] = {row, row * C.W_in, row * C.W_in * C.H_in,
                             row * C.W_in * C.H_in * static_cast<uint64_t>(C.cb_total)};
    const uint32_t box[5] = {kBK, static_cast<uint32_t>(bw * ew), static_cast<uint32_t>(bh * eh),
                             static_cast<uint32_t>(kd), 1};
    const uint32_t estr[5] = {1, static_cast<uint32_t>(ew), static_cast<uint32_t>(eh), 1, 1};
    if (!encode_bf16_tmap(&S.ma, C.a, 5, dims, str, box, estr)) return false;
  }
  {
    // weight [taps][ICp/64][OC][64] bf16
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(C.OC),
                              static_cast<uint64_t>(C.Kh * C.Kw) * icb};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(C.OC) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(oc_blk), static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&S.mb, C.b, 3, dims, str, box)) return false;
  }
  TcParams p{};
  p.mode = (direct ? 2 : 1) + (pixn ? 2 : 0);
  p.kd = kd;
  p.Nimg = static_cast<int>(C.N);
  p.OC = static_cast<int>(C.OC);
  p.out_ch = static_cast<int>(C.out_ch);
  p.Kh = static_cast<int>(C.Kh);
  p.Kw = static_cast<int>(C.Kw);
  p.H_out = static_cast<int>(C.H_out);
  p.W_out = static_cast<int>(C.W_out);
  p.sh = static_cast<int>(C.stride_h);
  p.sw = static_cast<int>(C.stride_w);
  p.pad_h = static_cast<int>(C.pad_h);
  p.pad_w = static_cast<int>(C.pad_w);
  p.dil_h = static_cast<int>(C.dil_h);
  p.dil_w = static_cast<int>(C.dil_w);
  p.gh = static_cast<int>(gcd64(C.dil_h, C.stride_h));
  p.gw = static_cast<int>(gcd64(C.dil_w, C.stride_w));
  p.tsh = static_cast<int>(C.stride_h / p.gh);
  p.tsw = static_cast<int>(C.stride_w / p.gw);
  p.dsh = static_cast<int>(C.dil_h / p.gh);
  p.dsw = static_cast<int>(C.dil_w / p.gw);
  p.invh = static_cast<int>(inv_mod(p.dsh, p.tsh));
  p.invw = static_cast<int>(inv_mod(p.dsw, p.tsw));
  p.osh = direct ? 1 : p.sh;
  p.osw = direct ? 1 : p.sw;
  p.ICp = static_cast<int>(C.ICp);
  p.icb = static_cast<int>(icb);
  p.BW = bw;
  p.BH = bh;
  p.tiles_w = static_cast<int>((Wq + bw - 1) / bw);
  p.tiles_h = static_cast<int>((Hq + bh - 1) / bh);
  p.tiles_oc = static_cast<int>((C.OC + oc_blk - 1) / oc_blk);
  const int64_t phases = direct ? 1 : C.stride_h;
  const int64_t units = phases * C.N * p.tiles_h * p.tiles_w * p.tiles_oc;
  if (units > (1ll << 30)) return false;
  p.total_units = static_cast<int>(units);
  p.subtiles = direct ? 1 : static_cast<int>(C.stride_w);
  // the most ring stages of any sub-tile (taps x channel-block stages)
  p.max_nstages = max_taps * static_cast<int>((icb + kd - 1) / kd);
  if (!direct && C.stride_h <= kMaxPhases) {
    // row phases with more taps first, so the heaviest units start earliest
    int order[kMaxPhases], taps[kMaxPhases];
    for (int ph = 0; ph < C.stride_h; ++ph) {
      taps[ph] = conv_t_phase_taps(ph, C.pad_h, C.stride_h, C.dil_h, C.Kh);
      order[ph] = ph;
    }
    std::stable_sort(order, order + C.stride_h, [&](int x, int y) { return taps[x] > taps[y]; });
    for (int i = 0; i < C.stride_h; ++i) p.ph_order[i] = static_cast<int8_t>(order[i]);
  }
  p.fd_oc = make_fastdiv(static_cast<uint32_t>(p.tiles_oc));
  p.fd_w = make_fastdiv(static_cast<uint32_t>(p.tiles_w));
  p.fd_h = make_fastdiv(static_cast<uint32_t>(p.tiles_h));
  p.fd_n = make_fastdiv(static_cast<uint32_t>(p.Nimg));
  p.phase_tab = 0;
  if (!direct && C.stride_h <= kMaxPhases && C.stride_w <= kMaxPhases) {
    // the first tap, tap count and first-tap input offset of each phase:
    // the least k >= 0 with k * dil = phase + pad (mod stride), k0 = ((t / g)
    // * inv) mod ts for t = (phase + pad) mod stride when g = gcd(dil,
    // stride) divides t (else no tap), and the input offset
    // (phase + pad - k0 * dil) / stride, an integer by construction
    auto fill = [](int nph, int pad, int stride, int dil, int K, int g, int ts, int inv, int* r0,
                   int* nt, int* d0) {
      for (int ph = 0; ph < nph; ++ph) {
        const int t = (ph + pad) % stride;
        r0[ph] = 0;
        nt[ph] = 0;
        d0[ph] = 0;
        if (t % g != 0) continue;
        const int k0 = static_cast<int>((static_cast<int64_t>(t / g) * inv) % ts);
        r0[ph] = k0;
        nt[ph] = k0 < K ? (K - k0 + ts - 1) / ts : 0;
        d0[ph] = (ph + pad - k0 * dil) / stride;
      }
    };
    fill(p.sh, p.pad_h, p.sh, p.dil_h, p.Kh, p.gh, p.tsh, p.invh, p.ph_r, p.ph_nt, p.ph_d0);
    fill(p.sw, p.pad_w, p.sw, p.dil_w, p.Kw, p.gw, p.tsw, p.invw, p.pw_r, p.pw_nt, p.pw_d0);
    p.phase_tab = 1;
  }
  p.ws = C.ws;
  p.bias = C.bias;
  p.rq = C.rq;
  p.out = C.out;
  p.acc_out = C.acc_out;
  p.store_mode = 0;
  p.a_bound_dev = nullptr;
  p.a_bound_host = C.a_bound;
  p.w_bound_dev = C.w_bound;
  // Output stores.  Register staging (2): each thread keeps its pixel's
  // earlier column phases and writes osw consecutive bytes per channel at the
  // unit's last phase (osw <= 2, aligned); otherwise one byte per output.
  const bool regstage = !pixn && C.out != nullptr && C.acc_out == nullptr && bn <= 128 &&
                        (p.osw == 1 || p.osw == 2) && C.W_out % p.osw == 0 &&
                        reinterpret_cast<uintptr_t>(C.out) % p.osw == 0;
  p.staged = regstage ? 2 : 0;
  S.p = p;
  S.bn = bn;
  S.kd = kd;
  S.pixn = pixn;
  S.single = p.max_nstages <= host_chunk_stages(C.a_bound, C.w_bound_host, kd);
  return true;
}

}  // namespace q8
