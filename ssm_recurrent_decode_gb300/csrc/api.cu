// api.cu -- the C ABI of libgdn_decode.so: host-side argument checks and kernel dispatch.
// Nothing here allocates, synchronises or touches device memory; every check runs on the host
// before the first CUDA call, and a rejected call launches nothing.
#include <cstdint>
#include <cmath>
#include <cstring>

#include "gdn_front.h"
#include "gdn_gemv.h"
#include "gdn_launch.h"
#include "mamba_decode.h"

namespace {

constexpr int kAbiVersion = 7;

bool k_supported(int K) { return K == 16 || K == 32 || K == 64 || K == 128; }
bool dtype_ok(int d) { return d == GDN_F32 || d == GDN_BF16; }
size_t dtype_size(int d) { return d == GDN_BF16 ? 2 : 4; }
bool aligned(const void *p, size_t bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

// Checks shared by every entry point that takes gdn_step_args.
int check_step(const gdn_step_args *a, bool indexed)
{
    if (!a) return GDN_ERR_NULL;
    if (a->B < 0 || a->H < 1 || a->HV < 1 || a->num_slots < 1) return GDN_ERR_SHAPE;
    if (a->HV % a->H != 0) return GDN_ERR_SHAPE;
    if (!k_supported(a->K) || a->V < 1 || a->V > 1024) return GDN_ERR_SHAPE;
    if ((int64_t)a->B * a->HV > INT32_MAX) return GDN_ERR_SHAPE;
    if (!indexed && a->num_slots < a->B) return GDN_ERR_SHAPE;
    if (!dtype_ok(a->in_dtype) || !dtype_ok(a->out_dtype) || !dtype_ok(a->state_dtype)) return GDN_ERR_DTYPE;
    if (a->gate_mode != GDN_GATE_RAW && a->gate_mode != GDN_GATE_DIRECT) return GDN_ERR_ARG;
    if (a->B == 0) return GDN_OK;
    if (!a->q || !a->k || !a->v || !a->state || !a->out) return GDN_ERR_NULL;
    if (a->gate_mode == GDN_GATE_RAW && (!a->a || !a->b || !a->A_log || !a->dt_bias)) return GDN_ERR_NULL;
    if (a->gate_mode == GDN_GATE_DIRECT && (!a->g || !a->beta)) return GDN_ERR_NULL;
    const size_t es = dtype_size(a->in_dtype);
    // q and k are read four elements at a time
    if (!aligned(a->q, 4 * es) || !aligned(a->k, 4 * es)) return GDN_ERR_ALIGN;
    if (a->q_stride % 4 != 0 || a->k_stride % 4 != 0) return GDN_ERR_ALIGN;
    if (!aligned(a->v, es) || !aligned(a->out, dtype_size(a->out_dtype))) return GDN_ERR_ALIGN;
    if (a->q_stride < (int64_t)a->H * a->K || a->k_stride < (int64_t)a->H * a->K ||
        a->v_stride < (int64_t)a->HV * a->V)
        return GDN_ERR_SHAPE;
    if (!aligned(a->state, 16)) return GDN_ERR_ALIGN;
    if (a->gate_mode == GDN_GATE_RAW && (!aligned(a->a, es) || !aligned(a->b, es))) return GDN_ERR_ALIGN;
    return GDN_OK;
}

gdn::StepLaunch make_step(const gdn_step_args *a, const int32_t *idx, int32_t pad)
{
    gdn::StepLaunch p;
    std::memset(&p, 0, sizeof(p));
    p.a = *a;
    p.idx = idx;
    p.pad = pad;
    p.G = a->HV / a->H;
    p.scale = a->scale != 0.f ? a->scale : 1.0f / std::sqrt((float)a->K);
    return p;
}

}  // namespace

namespace gdn {

// Host checks of gdn_decode_fused and the choice of kernel, without any CUDA launch.
int prepare_fused(const gdn_fused_args *a, FusedPlan *plan)
{
    plan->empty = false;
    plan->use_pipe = false;
    plan->sd = false;
    if (!a) return GDN_ERR_NULL;
    if (a->T < 0 || a->heads < 1 || a->num_slots < 1) return GDN_ERR_SHAPE;
    if (!k_supported(a->head_dim)) return GDN_ERR_SHAPE;
    if ((int64_t)a->T * a->heads > INT32_MAX) return GDN_ERR_SHAPE;
    if (a->gate_kind != GDN_FUSED_GATE_KDA && a->gate_kind != GDN_FUSED_GATE_GDN) return GDN_ERR_ARG;
    if (a->kda_gate_form != 0 && a->kda_gate_form != 1) return GDN_ERR_ARG;
    if (a->gate_act != GDN_ACT_SILU && a->gate_act != GDN_ACT_SIGMOID) return GDN_ERR_ARG;
    if (a->T == 0) {
        plan->empty = true;
        return GDN_OK;
    }
    if (!a->x || !a->conv_w || !a->conv_state || !a->raw_g || !a->raw_beta || !a->A_log ||
        !a->dt_bias || !a->state || !a->state_indices || !a->out_gate || !a->norm_w || !a->out)
        return GDN_ERR_NULL;
    const int64_t dim = (int64_t)a->heads * a->head_dim;
    if (a->x_stride < 3 * dim) return GDN_ERR_SHAPE;
    // row strides of the per-token inputs (0: dense)
    const int64_t g_width = a->gate_kind == GDN_FUSED_GATE_KDA ? dim : a->heads;
    const int64_t g_stride = a->raw_g_stride ? a->raw_g_stride : g_width;
    const int64_t b_stride = a->raw_beta_stride ? a->raw_beta_stride : a->heads;
    const int64_t og_stride = a->out_gate_stride ? a->out_gate_stride : dim;
    if (g_stride < g_width || b_stride < a->heads || og_stride < dim) return GDN_ERR_SHAPE;
    if (!aligned(a->x, 2) || !aligned(a->conv_state, 2) || !aligned(a->raw_g, 2) ||
        !aligned(a->raw_beta, 2) || !aligned(a->out_gate, 2) || !aligned(a->out, 2))
        return GDN_ERR_ALIGN;
    if (!aligned(a->conv_w, 16) || !aligned(a->state, 16) || !aligned(a->A_log, 4) ||
        !aligned(a->dt_bias, 4) || !aligned(a->norm_w, 4) || (a->conv_b && !aligned(a->conv_b, 4)))
        return GDN_ERR_ALIGN;
    if (a->kernel < GDN_KERNEL_AUTO || a->kernel > GDN_KERNEL_STAGE) return GDN_ERR_ARG;
    gdn::FusedLaunch &p = plan->p;
    std::memset(&p, 0, sizeof(p));
    p.a = *a;
    p.a.raw_g_stride = g_stride;
    p.a.raw_beta_stride = b_stride;
    p.a.out_gate_stride = og_stride;
    p.scale = a->scale != 0.f ? a->scale : 1.0f / std::sqrt((float)a->head_dim);
    // the pipelined kernel: head_dim 128, conv state in the DS ([slot][chan][tap]) or SD
    // ([slot][tap][chan]) layout, every bulk-copied row 16-byte aligned
    const bool ds = a->cs_stride_chan == 3 && a->cs_stride_tap == 1;
    const bool sd = a->cs_stride_chan == 1 && a->cs_stride_tap == 3 * dim;
    bool pipe_ok = a->head_dim == 128 && (ds || sd);
    const bool pipe_aligned = aligned(a->x, 16) && a->x_stride % 8 == 0 && aligned(a->conv_state, 16) &&
                              a->cs_stride_slot % 8 == 0 && aligned(a->raw_g, 16) && aligned(a->out_gate, 16) &&
                              og_stride % 8 == 0 && (a->gate_kind != GDN_FUSED_GATE_KDA || g_stride % 8 == 0) &&
                              aligned(a->dt_bias, 16) && aligned(a->state, 16);
    int sms = 0;
    if (pipe_ok) {
        int dev = 0, max_smem = 0;
        pipe_ok = cudaGetDevice(&dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
                  gdn::fused_pipe_fits(max_smem) &&
                  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    }
    // With at most two tiles per SM the persistent kernel's pipeline never fills and the per-tile
    // kernel was faster on GB300 (6.6 against 7.3 us for 96 tiles, 8.7 against 9.8 for 192); from
    // four tiles per SM the pipelined kernel wins.
    const bool few_tiles = (int64_t)a->T * a->heads <= 2 * (int64_t)sms;
    bool use_pipe = pipe_ok && pipe_aligned && !few_tiles;
    // From twelve tiles per SM one CTA per tile staged in shared memory beat the persistent kernel
    // (T = 128: 243.8 against 267.4 us; T = 32, 20 tiles per SM: 65.9 against 68.3; T = 24: 51.7
    // against 52.4; T = 20, 12.6 per SM: 44.1 against 44.4); at ten and five per SM it lost
    // (T = 16: 37.2 against 35.3; T = 8: 22.5 against 20.4).
    bool use_stage = use_pipe && (int64_t)a->T * a->heads >= 12 * (int64_t)sms;
    if (a->kernel == GDN_KERNEL_PIPE || a->kernel == GDN_KERNEL_STAGE) {
        if (!pipe_ok) return GDN_ERR_SHAPE;
        if (!pipe_aligned) return GDN_ERR_ALIGN;
        use_pipe = true;
        use_stage = a->kernel == GDN_KERNEL_STAGE;
    } else if (a->kernel == GDN_KERNEL_TILE) {
        use_pipe = use_stage = false;
    }
    plan->use_pipe = use_pipe;
    plan->use_stage = use_stage;
    plan->sd = sd;
    return GDN_OK;
}

int launch_fused_plan(const FusedPlan &plan, cudaStream_t stream, bool chained)
{
    if (plan.empty) return GDN_OK;
    if (plan.use_stage) return launch_fused_stage(plan.p, plan.sd, stream, chained);
    if (plan.use_pipe) return launch_fused_pipe(plan.p, plan.sd, stream, chained);
    return launch_fused(plan.p, stream, chained);
}

}  // namespace gdn

extern "C" {

int gdn_decode_step(const gdn_step_args *args, gdn_stream_t stream)
{
    int rc = check_step(args, false);
    if (rc != GDN_OK || args->B == 0) return rc;
    return gdn::launch_step(make_step(args, nullptr, 0), reinterpret_cast<cudaStream_t>(stream));
}

int gdn_decode_step_indexed(const gdn_step_args *args, const int32_t *cache_indices,
                            int32_t pad_slot_id, gdn_stream_t stream)
{
    int rc = check_step(args, true);
    if (rc != GDN_OK || args->B == 0) return rc;
    if (!cache_indices) return GDN_ERR_NULL;
    return gdn::launch_step(make_step(args, cache_indices, pad_slot_id),
                            reinterpret_cast<cudaStream_t>(stream));
}

int gdn_decode_step_indexed_chained(const gdn_step_args *args, const int32_t *cache_indices,
                                    int32_t pad_slot_id, gdn_stream_t stream)
{
    int rc = check_step(args, true);
    if (rc != GDN_OK || args->B == 0) return rc;
    if (!cache_indices) return GDN_ERR_NULL;
    return gdn::launch_step(make_step(args, cache_indices, pad_slot_id),
                            reinterpret_cast<cudaStream_t>(stream), true);
}

int gdn_decode_buffered(const gdn_step_args *args, const int32_t *cache_indices,
                        int32_t pad_slot_id, const gdn_ring_args *ring, gdn_stream_t stream)
{
    int rc = check_step(args, cache_indices != nullptr);
    if (rc != GDN_OK) return rc;
    if (args->state_dtype != GDN_F32) return GDN_ERR_DTYPE;
    if (!ring) return GDN_ERR_NULL;
    if (ring->L < 1 || ring->L > 64) return GDN_ERR_ARG;
    if (!dtype_ok(ring->ring_dtype)) return GDN_ERR_DTYPE;
    if (args->B == 0) return GDN_OK;
    if (!ring->d_cache || !ring->k_cache || !ring->g_cache || !ring->write_pos) return GDN_ERR_NULL;
    if (!aligned(ring->k_cache, 4 * dtype_size(ring->ring_dtype)) ||
        !aligned(ring->d_cache, dtype_size(ring->ring_dtype)) || !aligned(ring->g_cache, 4))
        return GDN_ERR_ALIGN;
    if (ring->kernel < GDN_KERNEL_AUTO || ring->kernel > GDN_KERNEL_STAGE) return GDN_ERR_ARG;
    const bool tile_ok = gdn::buffered_smem_bytes(ring->L, args->V, args->K) <= 200 * 1024;
    bool pipe_ok = args->K == 128 && args->V == 128 && (ring->L == 1 || ring->L % 4 == 0);
    const size_t es = dtype_size(args->in_dtype);
    const bool pipe_aligned =
        aligned(args->q, 16) && aligned(args->k, 16) && aligned(args->v, 16) &&
        (args->q_stride * (int64_t)es) % 16 == 0 && (args->k_stride * (int64_t)es) % 16 == 0 &&
        (args->v_stride * (int64_t)es) % 16 == 0 && aligned(ring->d_cache, 16) && aligned(ring->k_cache, 16) &&
        aligned(ring->g_cache, 16);
    int sms = 0;
    if (pipe_ok) {
        int dev = 0, max_smem = 0;
        pipe_ok = cudaGetDevice(&dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
                  gdn::buffered_pipe_fits(ring->L, args->in_dtype, ring->ring_dtype, max_smem) &&
                  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    }
    bool use_pipe, use_stage = false;
    if (ring->kernel == GDN_KERNEL_PIPE || ring->kernel == GDN_KERNEL_STAGE) {
        if (!pipe_ok) return GDN_ERR_SHAPE;
        if (!pipe_aligned) return GDN_ERR_ALIGN;
        use_pipe = true;
        use_stage = ring->kernel == GDN_KERNEL_STAGE;
    } else if (ring->kernel == GDN_KERNEL_TILE) {
        if (!tile_ok) return GDN_ERR_SHAPE;
        use_pipe = false;
    } else {
        // At L = 1 every step flushes and the per-tile kernel was faster on GB300 (170.4 against
        // 174.4 us at B = 256); from L = 8 the pipelined kernel is far ahead (96 against 147 us).
        // One CTA per tile staged in shared memory (GDN_KERNEL_STAGE) measured the same as the
        // persistent kernel (B = 256: 96.2 against 95.1 us at L = 16, 95.5 against 96.0 at L = 8), so
        // the persistent kernel stays the default.
        use_pipe = pipe_ok && pipe_aligned && !(ring->L == 1 && tile_ok);
        if (!use_pipe && !tile_ok) return GDN_ERR_SHAPE;
    }
    gdn::StepLaunch p = make_step(args, cache_indices, pad_slot_id);
    p.L = ring->L;
    p.d_cache = ring->d_cache;
    p.k_cache = ring->k_cache;
    p.g_cache = ring->g_cache;
    p.write_pos = ring->write_pos;
    if (use_stage) return gdn::launch_buffered_stage(p, ring->ring_dtype, reinterpret_cast<cudaStream_t>(stream));
    if (use_pipe) return gdn::launch_buffered_pipe(p, ring->ring_dtype, reinterpret_cast<cudaStream_t>(stream));
    return gdn::launch_buffered(p, ring->ring_dtype, reinterpret_cast<cudaStream_t>(stream));
}

int gdn_decode_fused(const gdn_fused_args *a, gdn_stream_t stream)
{
    gdn::FusedPlan plan;
    const int rc = gdn::prepare_fused(a, &plan);
    if (rc != GDN_OK) return rc;
    return gdn::launch_fused_plan(plan, reinterpret_cast<cudaStream_t>(stream));
}

const char *gdn_strerror(int status)
{
    switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_NULL: return "a required pointer is NULL";
    case GDN_ERR_SHAPE: return "unsupported or inconsistent size";
    case GDN_ERR_DTYPE: return "unsupported dtype";
    case GDN_ERR_ALIGN: return "a pointer or stride breaks the alignment rule";
    case GDN_ERR_LAUNCH: return "the CUDA launch failed";
    case GDN_ERR_ARG: return "invalid argument";
    case GDN_ERR_SCRATCH: return "the call needs more scratch than the fixed no-allocation buffer holds";
    default: return "unknown status";
    }
}

size_t gdn_abi_struct_size(int which)
{
    switch (which) {
    case 0: return sizeof(gdn_step_args);
    case 1: return sizeof(gdn_ring_args);
    case 2: return sizeof(gdn_fused_args);
    case 3: return sizeof(gdn_gemv_args);
    case 4: return sizeof(gdn_front_args);
    case 5: return sizeof(mamba_decode_args);
    default: return 0;
    }
}

int gdn_abi_version(void) { return kAbiVersion; }

}  // extern "C"
