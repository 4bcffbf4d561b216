// gq_pack.cu -- lossless repacking of canonical (GGUF-order) blocks into the
// planar layout the matvec kernels stream, and its exact inverse.
//
// "Gemma 4 M4 Max kernel roadmap", K4: the next axis considered there is a
// lossless fixed-shape Q4_0 repacking; requantization into a different
// native format is not permitted.  The packing here keeps every bit of
// every block (scales unchanged, codes permuted or XOR-ed), and the byte
// count is the same as the canonical blocks.
//
// Packed layouts (rows x K, nb = K/32 blocks, ns = K/256 super-blocks):
//   Q4_0: [rows*nb x 16 B nibbles, element order] [rows*nb x fp16 d]
//   Q8_0: [rows*nb x 32 B, byte = q XOR 0x80]     [rows*nb x fp16 d]
//   Q4_K: [rows*ns x 128 B, sub-block s at 16 s, element order]
//         [rows*ns x 16 B {d, dmin, 12 scale bytes}]
//   Q6_K: [rows*ns x 128 B low 4 code bits, element order]
//         [rows*ns x 64 B top 2 code bits: 32-bit word g holds the 16
//          elements 16g..16g+15; element 16g + 4a + i (a, i = 0..3) at
//          bits 4i + {0, 2, 16, 18}[a], +1]
//         [rows*ns x 16 B int8 sub-scales] [rows*ns x fp16 d]
// "Element order" means byte i of a 32-element group holds element 2i in
// its low nibble and element 2i+1 in its high nibble.
#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {

// canonical Q4_0 payload (byte j: element j low, j+16 high) -> element order
__device__ __forceinline__ void q4_canon_to_seq(const uint8_t *qs, uint8_t *out16)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e0 = 2 * i, e1 = 2 * i + 1;
        const int v0 = (e0 < 16) ? (qs[e0] & 15) : (qs[e0 - 16] >> 4);
        const int v1 = (e1 < 16) ? (qs[e1] & 15) : (qs[e1 - 16] >> 4);
        out16[i] = static_cast<uint8_t>(v0 | (v1 << 4));
    }
}
__device__ __forceinline__ void q4_seq_to_canon(const uint8_t *seq, uint8_t *qs)
{
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int lo = (j & 1) ? (seq[j >> 1] >> 4) : (seq[j >> 1] & 15);            // element j
        const int e = j + 16;
        const int hi = (e & 1) ? (seq[e >> 1] >> 4) : (seq[e >> 1] & 15);            // element j+16
        qs[j] = static_cast<uint8_t>(lo | (hi << 4));
    }
}

__global__ void k_pack_q4_0(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, long long nblk,
                            bool unpack)
{
    uint8_t *nib = dst;
    uint8_t *dsc = dst + nblk * 16;
    const uint8_t *pnib = src;
    const uint8_t *pdsc = src + nblk * 16;
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblk;
         b += (long long)gridDim.x * blockDim.x) {
        uint8_t tmp[16];
        if (!unpack) {
            const uint8_t *blk = src + b * 18;
            uint8_t qs[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) qs[j] = blk[2 + j];
            q4_canon_to_seq(qs, tmp);
#pragma unroll
            for (int j = 0; j < 16; ++j) nib[b * 16 + j] = tmp[j];
            dsc[b * 2] = blk[0];
            dsc[b * 2 + 1] = blk[1];
        } else {
            uint8_t seq[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) seq[j] = pnib[b * 16 + j];
            q4_seq_to_canon(seq, tmp);
            uint8_t *blk = dst + b * 18;
            blk[0] = pdsc[b * 2];
            blk[1] = pdsc[b * 2 + 1];
#pragma unroll
            for (int j = 0; j < 16; ++j) blk[2 + j] = tmp[j];
        }
    }
    // The decode kernels read their weights before they wait for the preceding kernel
    // (weights are model constants): make the packed bytes visible before this block exits.
    __threadfence();
}

__global__ void k_pack_q8_0(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, long long nblk,
                            bool unpack)
{
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblk;
         b += (long long)gridDim.x * blockDim.x) {
        if (!unpack) {
            const uint8_t *blk = src + b * 34;
            uint8_t *q = dst + b * 32;
            uint8_t *d = dst + nblk * 32 + b * 2;
            d[0] = blk[0];
            d[1] = blk[1];
#pragma unroll
            for (int j = 0; j < 32; ++j) q[j] = blk[2 + j] ^ 0x80u;
        } else {
            const uint8_t *q = src + b * 32;
            const uint8_t *d = src + nblk * 32 + b * 2;
            uint8_t *blk = dst + b * 34;
            blk[0] = d[0];
            blk[1] = d[1];
#pragma unroll
            for (int j = 0; j < 32; ++j) blk[2 + j] = q[j] ^ 0x80u;
        }
    }
    // The decode kernels read their weights before they wait for the preceding kernel
    // (weights are model constants): make the packed bytes visible before this block exits.
    __threadfence();
}

__global__ void k_pack_q4_k(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, long long nsup,
                            bool unpack)
{
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nsup;
         b += (long long)gridDim.x * blockDim.x) {
        if (!unpack) {
            const uint8_t *blk = src + b * 144;
            uint8_t *nib = dst + b * 128;
            uint8_t *rec = dst + nsup * 128 + b * 16;
            for (int j = 0; j < 16; ++j) rec[j] = blk[j];
            const uint8_t *qs = blk + 16;
            for (int s = 0; s < 8; ++s) {
                const uint8_t *chunk = qs + 32 * (s >> 1);
                for (int i = 0; i < 16; ++i) {
                    const int l0 = 2 * i, l1 = 2 * i + 1;
                    const int v0 = (s & 1) ? (chunk[l0] >> 4) : (chunk[l0] & 15);
                    const int v1 = (s & 1) ? (chunk[l1] >> 4) : (chunk[l1] & 15);
                    nib[16 * s + i] = static_cast<uint8_t>(v0 | (v1 << 4));
                }
            }
        } else {
            const uint8_t *nib = src + b * 128;
            const uint8_t *rec = src + nsup * 128 + b * 16;
            uint8_t *blk = dst + b * 144;
            for (int j = 0; j < 16; ++j) blk[j] = rec[j];
            uint8_t *qs = blk + 16;
            for (int c = 0; c < 4; ++c) {
                for (int l = 0; l < 32; ++l) {
                    const uint8_t lo_b = nib[16 * (2 * c) + (l >> 1)];
                    const uint8_t hi_b = nib[16 * (2 * c + 1) + (l >> 1)];
                    const int lo = (l & 1) ? (lo_b >> 4) : (lo_b & 15);
                    const int hi = (l & 1) ? (hi_b >> 4) : (hi_b & 15);
                    qs[32 * c + l] = static_cast<uint8_t>(lo | (hi << 4));
                }
            }
        }
    }
    // The decode kernels read their weights before they wait for the preceding kernel
    // (weights are model constants): make the packed bytes visible before this block exits.
    __threadfence();
}

// Q6_K canonical block (ql[128], qh[64], sc[16], d): in each 128-weight half
// h, weight 32c + l has its low bits in ql[64h + l + 32(c % 2)] (low nibble
// for c < 2, high nibble otherwise) and its top bits at bit 2c of qh[32h + l].
// Packed top bits: bit position of element e's pair within its 32-bit word
// (word e / 16): quarter a = (e / 4) % 4 of the 16 elements sits at offset
// {0, 2, 16, 18}[a], element i = e % 4 of the quarter 4i above it.  Shifted
// by {+4, +2, -12, -14}[a], every pair of a quarter lands at bits 4i + 4,
// just above its element's nibble in the low-bit word (the matvec joins the
// two with one bit-select per two elements).
__device__ __forceinline__ int q6_top_bit(int e)
{
    const int a = (e >> 2) & 3;
    return 4 * (e & 3) + ((a & 1) ? 2 : 0) + ((a & 2) ? 16 : 0);
}

__global__ void k_pack_q6_k(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, long long nsup,
                            bool unpack)
{
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nsup;
         b += (long long)gridDim.x * blockDim.x) {
        if (!unpack) {
            const uint8_t *blk = src + b * 210;
            uint8_t *lo = dst + b * 128;
            uint32_t hw[16];
            uint8_t *sc = dst + nsup * 192 + b * 16;
            uint8_t *dd = dst + nsup * 208 + b * 2;
            for (int j = 0; j < 16; ++j) sc[j] = blk[192 + j];
            dd[0] = blk[208];
            dd[1] = blk[209];
            for (int i = 0; i < 128; ++i) lo[i] = 0;
            for (int i = 0; i < 16; ++i) hw[i] = 0u;
            for (int e = 0; e < 256; ++e) {
                const int h = e >> 7, c = (e >> 5) & 3, l = e & 31;
                const uint8_t qlb = blk[64 * h + l + 32 * (c & 1)];
                const int q_lo = (c < 2) ? (qlb & 15) : (qlb >> 4);
                const uint32_t q_hi = (blk[128 + 32 * h + l] >> (2 * c)) & 3;
                lo[e >> 1] |= static_cast<uint8_t>(q_lo << (4 * (e & 1)));
                hw[e >> 4] |= q_hi << q6_top_bit(e & 15);
            }
            uint8_t *hi = dst + nsup * 128 + b * 64;
            for (int i = 0; i < 64; ++i) hi[i] = static_cast<uint8_t>(hw[i >> 2] >> (8 * (i & 3)));
        } else {
            const uint8_t *lo = src + b * 128;
            const uint8_t *hi = src + nsup * 128 + b * 64;
            const uint8_t *sc = src + nsup * 192 + b * 16;
            const uint8_t *dd = src + nsup * 208 + b * 2;
            uint8_t *blk = dst + b * 210;
            for (int j = 0; j < 16; ++j) blk[192 + j] = sc[j];
            blk[208] = dd[0];
            blk[209] = dd[1];
            for (int i = 0; i < 192; ++i) blk[i] = 0;
            for (int e = 0; e < 256; ++e) {
                const int h = e >> 7, c = (e >> 5) & 3, l = e & 31;
                const int q_lo = (lo[e >> 1] >> (4 * (e & 1))) & 15;
                const int g = e >> 4, p = q6_top_bit(e & 15);
                const int q_hi = (hi[4 * g + (p >> 3)] >> (p & 7)) & 3;
                blk[64 * h + l + 32 * (c & 1)] |= static_cast<uint8_t>(q_lo << ((c < 2) ? 0 : 4));
                blk[128 + 32 * h + l] |= static_cast<uint8_t>(q_hi << (2 * c));
            }
        }
    }
    // The decode kernels read their weights before they wait for the preceding kernel
    // (weights are model constants): make the packed bytes visible before this block exits.
    __threadfence();
}

int launch_pack(int format, const void *src, void *dst, int rows, int K, bool unpack, cudaStream_t s)
{
    const long long n = (format == GQ_FORMAT_Q4_K || format == GQ_FORMAT_Q6_K) ? (long long)rows * (K / 256)
                                                                               : (long long)rows * (K / 32);
    const int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    const long long cap = (long long)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const uint8_t *a = static_cast<const uint8_t *>(src);
    uint8_t *b = static_cast<uint8_t *>(dst);
    switch (format) {
    case GQ_FORMAT_Q4_0: k_pack_q4_0<<<(unsigned)blocks, threads, 0, s>>>(a, b, n, unpack); break;
    case GQ_FORMAT_Q8_0: k_pack_q8_0<<<(unsigned)blocks, threads, 0, s>>>(a, b, n, unpack); break;
    case GQ_FORMAT_Q4_K: k_pack_q4_k<<<(unsigned)blocks, threads, 0, s>>>(a, b, n, unpack); break;
    case GQ_FORMAT_Q6_K: k_pack_q6_k<<<(unsigned)blocks, threads, 0, s>>>(a, b, n, unpack); break;
    default: return GQ_ERR_FORMAT;
    }
    return status_from(cudaGetLastError());
}

}  // namespace gq
