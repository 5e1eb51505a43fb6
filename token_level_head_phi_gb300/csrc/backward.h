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
int launch_bwd_summary(const Plan& p, const BwdBuffers& w, const void* k, const void* v, void* dk, void* dv,
                       void* stream);

}  // namespace mhla
