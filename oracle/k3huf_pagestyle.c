/*
 * k3huf_pagestyle.c -- a second CPU decoder of the k3_huf container, in the
 * style of the article's own decoder, used only as the like-for-like CPU
 * timing beside the bit-serial oracle.
 *
 * TEST INFRASTRUCTURE, like the rest of this directory: only the test
 * suite and the benchmark's CPU-baseline leg call it.  It shares nothing
 * with the CUDA library.  From the oracle it uses only the canonical code
 * assignment (orc_canonical) and the header check (orc_layer_info); its
 * decode and its table are its own, and the tests pin both against the
 * oracle's bit-serial decoder.
 *
 * Source: the article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：一次被解码速度
 * 判死刑的 Huffman 压缩实验", sections 已实现的部分 (a 4096-entry table of
 * (symbol << 4) | length indexed by the next 12 bits), 规范码分配与 Kraft
 * 校验 (its closing paragraph on the decode loop: a bit accumulator whose
 * top holds the head of the stream, a refill that serves several symbols,
 * and the even bytes copied in a separate loop after the odd plane) and
 * 让方案被搁置的测量：解码速度 (that loop's speed, about 0.31 GB/s per
 * core).  The article decodes a stripe from its first bit to its last; the
 * chunk and sub-stream indexes of this container are not read (chunks
 * follow one another without gaps in the bit stream).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* from k3huf_oracle.c */
void orc_canonical(const int len[256], int maxlen, uint32_t count[33], uint32_t first[33], uint32_t code[256]);
int orc_layer_info(const uint8_t *blob, uint64_t bytes, uint64_t info[10]);

#define PS_WIN        12          /* table index bits (the format's code length limit) */
#define PS_OK          0
#define PS_E_ARG      -1
#define PS_E_FORMAT   -5

static uint64_t ps_get(const uint8_t *p, int n)
{
    uint64_t v = 0;
    for (int i = n - 1; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}

/* Table entry w = (symbol << 4) | length of the code that is a prefix of
 * the 12-bit window w, or 0 where no code is (an incomplete code).  The
 * codes are the canonical ones of codelen.  Returns PS_E_ARG for lengths
 * above 12. */
int orc_ps_build(const uint8_t codelen[256], uint16_t lut[1 << PS_WIN])
{
    int len[256];
    uint32_t count[33], first[33], code[256];
    for (int s = 0; s < 256; s++) {
        if (codelen[s] > PS_WIN) return PS_E_ARG;
        len[s] = codelen[s];
    }
    orc_canonical(len, PS_WIN, count, first, code);
    memset(lut, 0, sizeof(uint16_t) << PS_WIN);
    for (int s = 0; s < 256; s++) {
        if (!len[s]) continue;
        uint32_t base = code[s] << (PS_WIN - len[s]), span = 1u << (PS_WIN - len[s]);
        for (uint32_t j = 0; j < span; j++) lut[base + j] = (uint16_t)((s << 4) | len[s]);
    }
    return PS_OK;
}

/* Decode stripe s of a layer container: the odd plane into hi (the
 * stripe's n_values bytes, caller-owned), then the bf16 values into out at
 * the stripe's output offset.  Returns PS_OK, or PS_E_FORMAT for a window
 * that starts no code, a stream read past its recorded length, or a
 * malformed container. */
int orc_ps_decode_stripe(const uint8_t *blob, uint64_t bytes, uint32_t s, uint8_t *hi, uint8_t *out)
{
    uint64_t info[10];
    if (orc_layer_info(blob, bytes, info)) return PS_E_FORMAT;
    const uint64_t n_tables = info[1], n_tensors = info[2], n_stripes = info[3];
    if (s >= n_stripes) return PS_E_ARG;
    const uint8_t *e = blob + 64 + 256 * n_tables + 32 * n_tensors + 32ull * s;
    const uint64_t off = ps_get(e, 8), sbytes = ps_get(e + 8, 8), out_off = ps_get(e + 16, 8);
    const uint32_t table = (uint32_t)ps_get(e + 28, 4);
    if (table >= n_tables || off + sbytes > bytes) return PS_E_FORMAT;
    const uint8_t *st = blob + off;
    const uint64_t nv = ps_get(st + 8, 4), huff_bits = ps_get(st + 16, 8);
    const uint64_t bits_off = ps_get(st + 24, 4), even_off = ps_get(st + 28, 4);
    if (even_off + nv > sbytes || bits_off + (huff_bits + 7) / 8 > even_off) return PS_E_FORMAT;

    uint16_t lut[1 << PS_WIN];
    if (orc_ps_build(blob + 64 + 256ull * table, lut)) return PS_E_FORMAT;

    /* odd plane: the accumulator's top bits are the stream's next bits */
    const uint8_t *p = st + bits_off, *const pend = p + (huff_bits + 7) / 8;
    uint64_t acc = 0;
    int nb = 0;                                     /* valid bits in acc */
    for (uint64_t i = 0; i < nv; i++) {
        if (nb < PS_WIN) {                          /* refill whole bytes: one refill serves several codes */
            while (nb <= 56) {
                const uint64_t b = p < pend ? *p : 0u;
                p++;
                acc |= b << (56 - nb);
                nb += 8;
            }
        }
        const uint32_t ent = lut[acc >> (64 - PS_WIN)];
        const int l = (int)(ent & 15u);
        if (l == 0) return PS_E_FORMAT;
        hi[i] = (uint8_t)(ent >> 4);
        acc <<= l;
        nb -= l;
    }
    if ((uint64_t)(p - (st + bits_off)) * 8 - (uint64_t)nb > huff_bits) return PS_E_FORMAT;

    /* even plane, in a loop of its own (little-endian bf16: low byte first) */
    const uint8_t *even = st + even_off;
    uint8_t *o = out + out_off;
    for (uint64_t i = 0; i < nv; i++) {
        o[2 * i] = even[i];
        o[2 * i + 1] = hi[i];
    }
    return PS_OK;
}
