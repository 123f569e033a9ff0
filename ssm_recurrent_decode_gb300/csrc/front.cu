// front.cu -- gdn_decode_front: one DeltaNet layer's decode forward (input projection -> conv
// update, delta step, gated RMSNorm -> output projection) as three launches of this library's
// kernels on one stream, every stage checked on the host before the first launch.
//
// Source: "Optimization Log: Qwen3.5-27B Dense on B200", Integration (the DeltaNet forward of the
// model patcher: proj + conv1d + recurrent + norm_gated + output) and Kernel 3 (the projections).
#include <cstdint>

#include "gdn_front.h"
#include "gdn_gemv.h"
#include "gdn_launch.h"
#include "gemv_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int64_t gdn_front_proj_width(int32_t heads, int32_t head_dim, int32_t gate_kind)
{
    const int64_t dim = (int64_t)heads * head_dim;
    if (gate_kind == GDN_FUSED_GATE_KDA) return 4 * dim + dim + heads;
    if (gate_kind == GDN_FUSED_GATE_GDN) return 4 * dim + heads + heads;
    return 0;
}

int gdn_decode_front(const gdn_front_args *a, gdn_stream_t stream)
{
    if (!a) return GDN_ERR_NULL;
    const gdn_fused_args &c = a->core;
    if (a->T < 0 || a->hidden < 1 || a->hidden % 8 != 0 || c.heads < 1 || c.head_dim < 1) return GDN_ERR_SHAPE;
    if (a->in_splits < 0 || a->in_splits > gdn::kGemvMaxCluster || a->out_splits < 0 ||
        a->out_splits > gdn::kGemvMaxCluster)
        return GDN_ERR_ARG;
    const int64_t P = gdn_front_proj_width(c.heads, c.head_dim, c.gate_kind);
    if (P == 0) return GDN_ERR_ARG;
    const int64_t dim = (int64_t)c.heads * c.head_dim;
    const int64_t G = c.gate_kind == GDN_FUSED_GATE_KDA ? dim : c.heads;
    if (P > INT32_MAX) return GDN_ERR_SHAPE;
    if (a->T == 0) return GDN_OK;
    if (!a->z || !a->o) return GDN_ERR_NULL;
    if (!aligned16(a->z) || !aligned16(a->o)) return GDN_ERR_ALIGN;
    const auto *z = static_cast<const uint16_t *>(a->z);   // bf16 elements, addressed as 2 bytes

    // (1) z = x W_in^T
    gdn_gemv_args in = {};
    in.T = a->T;
    in.N = (int32_t)P;
    in.Kd = a->hidden;
    in.out_dtype = GDN_BF16;
    in.x = a->x;
    in.x_stride = a->x_stride;
    in.W = a->W_in;
    in.y = a->z;
    in.y_stride = P;
    in.splits = a->in_splits;
    in.err_flags = c.err_flags;
    // (2) o = conv -> step -> gated RMSNorm on views of z
    gdn_fused_args f = c;
    f.T = a->T;
    f.x = z;
    f.x_stride = P;
    f.out_gate = z + 3 * dim;
    f.out_gate_stride = P;
    f.raw_g = z + 4 * dim;
    f.raw_g_stride = P;
    f.raw_beta = z + 4 * dim + G;
    f.raw_beta_stride = P;
    f.out = a->o;
    // (3) y = o W_out^T
    gdn_gemv_args out = {};
    out.T = a->T;
    out.N = a->hidden;
    out.Kd = (int32_t)dim;
    out.out_dtype = a->y_dtype;
    out.x = a->o;
    out.x_stride = dim;
    out.W = a->W_out;
    out.y = a->y;
    out.y_stride = a->y_stride;
    out.splits = a->out_splits;
    out.err_flags = c.err_flags;

    int in_splits = 0, out_splits = 0, rc;
    gdn::FusedPlan plan;
    if ((rc = gdn::gemv_check(&in, &in_splits)) != GDN_OK) return rc;
    if ((rc = gdn::prepare_fused(&f, &plan)) != GDN_OK) return rc;
    if ((rc = gdn::gemv_check(&out, &out_splits)) != GDN_OK) return rc;
    if (in_splits > gdn::kGemvMaxCluster || out_splits > gdn::kGemvMaxCluster) return GDN_ERR_ARG;

    // The fused step and the output projection are chained launches: each may start while the
    // kernel before it finishes and waits for it before reading that kernel's output. The input
    // projection is an ordinary launch, so everything before this call has completed first.
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = gdn::gemv_launch(in, in_splits, s)) != GDN_OK) return rc;
    if ((rc = gdn::launch_fused_plan(plan, s, true)) != GDN_OK) return rc;
    return gdn::gemv_launch(out, out_splits, s, true);
}

}  // extern "C"
