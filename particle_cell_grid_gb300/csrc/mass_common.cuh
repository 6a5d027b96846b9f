// mass_common.cuh -- per-particle coefficient of the ECSIM mass matrix, shared
// by the first-order (mass_matrix.cu) and second-order (mass_tsc.cu) kernels.
//
// Pennati & Markidis, Sec. 2.1, Eqs. (5)-(6): s_p = w_p alpha_p with
//   alpha = (I - C(omega) + omega omega^T) / (1 + |omega|^2),  C(omega) u = omega x u,
// row-major s[3 i + j].
#pragma once

namespace pcg {

__device__ __forceinline__ void alpha_w(float w, float ox, float oy, float oz, float (&s)[9]) {
    const float n2 = ox * ox + oy * oy + oz * oz;
    const float f = w / (1.f + n2);
    s[0] = f * (1.f + ox * ox);
    s[1] = f * (oz + ox * oy);
    s[2] = f * (-oy + ox * oz);
    s[3] = f * (-oz + oy * ox);
    s[4] = f * (1.f + oy * oy);
    s[5] = f * (ox + oy * oz);
    s[6] = f * (oy + oz * ox);
    s[7] = f * (-ox + oz * oy);
    s[8] = f * (1.f + oz * oz);
}

}  // namespace pcg
