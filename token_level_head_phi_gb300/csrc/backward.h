// Interface between the host dispatcher and the backward kernels.
#pragma once

#include "plan.h"

namespace mhla {

// Float32 workspace of the backward pass (SIMT plan: Q = M * splits pieces).
struct BwdBuffers {
  const float* mc;     // [M][M]
  float* stack;        // [BH][Q][R] forward summaries per piece (S_b | z_b | v_b)
  float* mixed;        // [BH][M][R] forward mixed summaries
  float* rowsum;       // [M] sum_b Mc[i][b]
  float* dmixp;        // [BH][Q][R] per query piece: partial dS~ | dz~ | dv~
  float* dnp;          // [BH][Q] per query piece: partial dn~ (MALA)
  float* dstack;       // [BH][M][R] dS_b | dz_b | dv_b
  float* dmc;          // [M][M] output
  // causal form (nullptr otherwise)
  const float* diag;   // [BH][M] in-block term of dMc[i][i]; dMc above the diagonal is 0
  const float* xk;     // [BH][N][d] in-block part of dphi(k) (laid out like K, float32)
  const float* xv;     // [BH][N][d] in-block part of dv
  float* mc_partial;   // [groups][mc_heads][M][M] partial sums of dMc (bwd_mc_partial_bytes, may be 0)
};

// Buffers of the causal backward's in-block kernels (simt_causal_bwd.cu).
struct CausalBwdBuffers {
  const float* mc;            // the full Mc (its diagonal weighs the in-block terms)
  const float* mixed;         // [BH][M][R] Sp_i, zp_i, vp_i: earlier blocks through Mc's strict lower triangle
  const float* rowsum_lower;  // [M] row sums of Mc's strict lower triangle
  float* dmixp;               // [BH][M * splits][R] out: dSp_i, dzp_i, dvp_i in the block's first piece row
  float* dnp;                 // [BH][M * splits] out: dnp_i (MALA), likewise
  float* diag;                // [BH][M] out: in-block term of dMc[i][i]
  float* tokbuf;              // [BH][N][d + 4] scratch: dnum_t, ds_t, gamma_t (16-byte rows)
  float* xk;                  // [BH][N][d] out: in-block part of dphi(k)
  float* xv;                  // [BH][N][d] out: in-block part of dv
};

// The four steps of the float32 backward after the forward summaries and
// mixing (w.stack, w.mixed, w.rowsum) are in place, in this order:
//   output:  dq and per query piece the partial dS~, dz~, dv~ (w.dmixp), dn~ (w.dnp)
//   mix:     w.dstack = dS_b, dz_b, dv_b (Mc transposed times the partials)
//   mc:      w.dmc (summed over heads)
//   summary: dk, dv
int launch_bwd_output(const Plan& p, const BwdBuffers& w, const void* q, const void* dout, void* dq, void* stream);
int launch_bwd_mix(const Plan& p, const BwdBuffers& w, void* stream);
int launch_bwd_mc(const Plan& p, const BwdBuffers& w, void* stream);
// Workspace of the dMc partial sums (0 when one group covers every unit).
size_t bwd_mc_partial_bytes(const Plan& p);
int launch_bwd_summary(const Plan& p, const BwdBuffers& w, const void* k, const void* v, void* dk, void* dv,
                       void* stream);
// Causal form, after the forward summaries and the strict-lower mixing: dq,
// the prefix partials, dn~, the diagonal of dMc and the in-block parts of
// dphi(k), dv (then launch_bwd_mix with Mc's strict lower triangle,
// launch_bwd_mc and launch_bwd_summary with w.diag, w.xk, w.xv set).
int launch_bwd_causal_block(const Plan& p, const CausalBwdBuffers& c, const void* q, const void* k, const void* v,
                            const void* dout, void* dq, void* stream);

}  // namespace mhla
