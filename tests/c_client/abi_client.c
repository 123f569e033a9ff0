/*
 * abi_client.c -- a plain C (C11) client of libgdn_decode.so, built against the headers in
 * include/ only. It needs no GPU: it prints the library's ABI version, the argument struct sizes
 * as this C compiler lays them out next to the library's own, and the status codes that the
 * host-side checks return for calls that must be refused before any CUDA work (the device
 * addresses below are aligned and never dereferenced).
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn_decode.h"
#include "gdn_front.h"
#include "gdn_gemv.h"
#include "mamba_decode.h"

static gdn_step_args valid_step(void)
{
    const uintptr_t base = (uintptr_t)1 << 40;
    gdn_step_args s;
    memset(&s, 0, sizeof s);
    s.B = 4; s.H = 2; s.HV = 4; s.K = 128; s.V = 128; s.num_slots = 4;
    s.in_dtype = GDN_BF16; s.out_dtype = GDN_BF16;
    s.q = (const void *)base; s.k = (const void *)(base + 512); s.v = (const void *)(base + 1024);
    s.q_stride = s.k_stride = s.v_stride = 2 * 2 * 128 + 4 * 128;
    s.gate_mode = GDN_GATE_RAW;
    s.a = (const void *)(base + 4096); s.b = (const void *)(base + 8192);
    s.A_log = (const float *)(base + 12288); s.dt_bias = (const float *)(base + 16384);
    s.state = (void *)(base + ((uintptr_t)1 << 30)); s.out = (void *)(base + ((uintptr_t)1 << 31));
    return s;
}

int main(void)
{
    printf("version %d\n", gdn_abi_version());
    printf("c_sizes %zu %zu %zu %zu %zu %zu\n", sizeof(gdn_step_args), sizeof(gdn_ring_args),
           sizeof(gdn_fused_args), sizeof(gdn_gemv_args), sizeof(gdn_front_args), sizeof(mamba_decode_args));
    printf("lib_sizes %zu %zu %zu %zu %zu %zu\n", gdn_abi_struct_size(0), gdn_abi_struct_size(1),
           gdn_abi_struct_size(2), gdn_abi_struct_size(3), gdn_abi_struct_size(4), gdn_abi_struct_size(5));

    gdn_step_args s = valid_step();
    printf("null_args %d\n", gdn_decode_step(NULL, NULL));
    s.K = 96;
    printf("bad_K %d\n", gdn_decode_step(&s, NULL));
    s = valid_step();
    s.in_dtype = 7;
    printf("bad_dtype %d\n", gdn_decode_step(&s, NULL));
    s = valid_step();
    s.state = (void *)(((uintptr_t)1 << 40) + 8);
    printf("misaligned_state %d\n", gdn_decode_step(&s, NULL));
    s = valid_step();
    s.gate_mode = 5;
    printf("bad_gate_mode %d\n", gdn_decode_step(&s, NULL));
    s = valid_step();
    printf("null_indices %d\n", gdn_decode_step_indexed(&s, NULL, -1, NULL));
    s = valid_step();
    s.B = 0;
    printf("empty_batch %d\n", gdn_decode_step(&s, NULL));
    printf("front_width %lld\n", (long long)gdn_front_proj_width(32, 128, GDN_FUSED_GATE_GDN));
    printf("strerror_null %s\n", gdn_strerror(GDN_ERR_NULL));
    return 0;
}
