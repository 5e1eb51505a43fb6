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

// Called after each backward phase with its index (2: output step, 3:
// gradient mixing, 4: dMc, 5: dk and dv) and the stream.
using PhaseMark = void (*)(int phase, void* stream);

// dq, dk, dv (q's dtype) and w.dmc from the recomputed forward in w.
int launch_backward(const Plan& p, const BwdBuffers& w, const void* q, const void* k, const void* v,
                    const void* dout, void* dq, void* dk, void* dv, void* stream, PhaseMark mark);

}  // namespace mhla
