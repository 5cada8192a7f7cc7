/*
 * GAAC oracle: a plain, scalar, slow CPU statement of the GAAC codec and of
 * decode attention in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code, header, table or constant generator with the CUDA library; every
 * constant below is restated here from the format definition.
 *
 * Source of the method: "GAAC: Lossless KV Compression for Bandwidth-Efficient
 * LLM Inference on Personal Devices" (Guo, George, Joshi), summary page:
 *   - section 3.1 (Lossless KV Compression): per-head-channel calibrated
 *     exponent windows of length 8 and 16; groups of eight values use a 3-bit,
 *     4-bit or raw exponent mode depending on whether every offset fits; an
 *     out-of-window value widens the whole group; sign and mantissa are kept
 *     unchanged.
 *   - section 3.2 (Attention with On-the-Fly Decompression): compressed blocks
 *     and the raw tail share one softmax.
 *   - section 3.3 and Figure 3 (Block-Wise Compression Scheduling):
 *     fixed-capacity slots, oversized blocks stay BF16, BF16 tail filled and
 *     then finalized.
 *   - Appendix D, Table 9 (Storage): 3-bit exponent codes, 2-bit mode tags,
 *     escape bytes, fixed-capacity escape slots.
 * The page gives no bit layout.  This file fixes one, "GAAC tile format v3",
 * summarised below and spelled out rule by rule at the step that follows it.
 *
 * Format v3 in brief (all multi-byte fields little-endian):
 *   tile        64 tokens x 128 channels of one (sequence, block, kv-head, K|V)
 *   storage     K tiles: element (t,c) at s = t*128 + c   (token-major)
 *   order       V tiles: the operand order of storage_index below (a
 *               32-element unit holds 2 channels x 4 tokens of each of four
 *               16-channel blocks)
 *   group       8 consecutive elements in storage order, G = s / 8
 *   eighth      128 consecutive groups (1024 elements), w = G / 128
 *   slot image  [0,8192)      mantissa of element s in bits 0-6 of byte s; bit 7
 *                             of byte s holds the sign of element
 *                             4*(s/4) + (s+3)%4 (signs rotated by one byte
 *                             inside each aligned group of four)
 *               [8192,11264)  code plane: 3 words per 32-element unit
 *               [11264,11520) tag plane: 2 bits per group
 *               [11520,11536) escape directory: 8 u16; entry w = (4-bit groups
 *                             of eighths 0..w) | (raw groups of eighths 0..w) << 9
 *                             (each count modulo its field: 9 and 7 bits; exact
 *                             whenever the escape area fits 496 bytes)
 *               [11536,12032) escape area, capacity 496, zero filled: first one
 *                             byte per 4-bit group, then eight exponent bytes
 *                             per raw group, each in group order
 *   raw tile    8192 BF16 words in storage order
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_D 128               /* head_dim */
#define ORC_BLOCK 64            /* tokens per tile */
#define ORC_TILE 8192           /* elements per tile */
#define ORC_GROUPS 1024         /* groups of 8 per tile */
#define ORC_UNITS 256           /* 32-element code units per tile */
#define ORC_OFF_CODE 8192
#define ORC_OFF_TAG 11264
#define ORC_OFF_DIR 11520          /* escape directory: 8 x u16 */
#define ORC_OFF_ESC 11536          /* escape bytes */
#define ORC_ESC_CAP 496
#define ORC_DIR_GROUPS 128         /* groups per directory entry (an eighth of the tile) */
#define ORC_SLOT 12032

enum { ORC_KIND_K = 0, ORC_KIND_V = 1 };
enum { ORC_M3BIT = 0, ORC_M4BIT = 1, ORC_MRAW = 2 };

/* ---- BF16 fields (section 3.1: sign and mantissa verbatim, exponent coded) */
static unsigned bf16_exponent(uint16_t x) { return (x >> 7) & 0xFFu; }
static unsigned bf16_signmant(uint16_t x) { return ((x >> 8) & 0x80u) | (x & 0x7Fu); }
static uint16_t bf16_join(unsigned signmant, unsigned exponent) {
    return (uint16_t)(((signmant & 0x80u) << 8) | ((exponent & 0xFFu) << 7) | (signmant & 0x7Fu));
}

/* ---- sign|mantissa plane (format v3, as v2): byte s keeps the mantissa of element s
 * and the sign of element sign_source(s), the previous element of the same
 * aligned group of four, cyclically (byte 4i holds the sign of 4i+3). */
static int sign_source(int s) { return 4 * (s / 4) + (s + 3) % 4; }
static int sign_holder(int s) { return 4 * (s / 4) + (s + 1) % 4; }

/* ---- storage order of a tile (format v3)
 * K: token-major, s = t*128 + c.
 * V: s = 1024*(2*w + h) + 32*(4*g + q) + 8*i + r with
 *      w = t / 16            (quarter of the block's tokens)
 *      q = (t % 8) / 2,  r bit 1 = t % 2,  r bit 2 = (t % 16) / 8
 *      h = c / 64,  i = (c / 16) % 4,  g = c % 8,  r bit 0 = (c % 16) / 8
 * so that unit 32*(2w+h) + 4g + q holds, for the four 16-channel blocks
 * 4h..4h+3, channels 16m+g and 16m+g+8 at tokens 16w + 2q + {0,1,8,9}: the
 * elements one lane of a 16x16 operand tile of a tensor-core product over
 * (channels x tokens) holds.  A group (r = 0..7) is two channels x four tokens. */
int gaac_ref_storage_index(int kind, int t, int c) {
    if (kind == ORC_KIND_K) return t * ORC_D + c;
    int w = t / 16, q = (t % 8) / 2, h = c / 64, i = (c / 16) % 4, g = c % 8;
    int r = (c % 16) / 8 + 2 * (t % 2) + 4 * ((t % 16) / 8);
    return 1024 * (2 * w + h) + 32 * (4 * g + q) + 8 * i + r;
}
static void storage_to_tc(int kind, int s, int* t, int* c) {
    if (kind == ORC_KIND_K) { *t = s / ORC_D; *c = s % ORC_D; return; }
    int u = s / 32, j = s % 32, eighth = u / 32, lane = u % 32;
    int w = eighth / 2, h = eighth % 2, g = lane / 4, q = lane % 4, i = j / 8, r = j % 8;
    *t = 16 * w + 8 * (r >> 2) + 2 * q + ((r >> 1) & 1);
    *c = 16 * (4 * h + i) + 8 * (r & 1) + g;
}
static int channel_of(int kind, int s) { int t, c; storage_to_tc(kind, s, &t, &c); return c; }

/* ---- calibration (section 3.1 and 4.7.1: windows of 8 and 16 exponents per
 * head-channel, chosen from calibration data).  Window with the largest count;
 * ties go to the smallest base. */
static int best_window_n(const uint64_t* hist, int nbins, int width) {
    uint64_t best = 0;
    int arg = 0;
    int have = 0;
    for (int b = 0; b + width <= nbins; ++b) {
        uint64_t sum = 0;
        for (int i = 0; i < width; ++i) sum += hist[b + i];
        if (!have || sum > best) { best = sum; arg = b; have = 1; }
    }
    return arg;
}

static int best_window(const uint64_t* hist, int width) { return best_window_n(hist, 256, width); }
int gaac_ref_best_window(const uint64_t* hist, int width) { return best_window(hist, width); }

/* x[t*tok_stride + h*128 + c] for t < n_tok; writes base3[h*128+c], base4[h*128+c]. */
void gaac_ref_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_heads,
                        uint8_t* base3, uint8_t* base4) {
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < ORC_D; ++c) {
            uint64_t hist[256];
            memset(hist, 0, sizeof hist);
            for (int64_t t = 0; t < n_tok; ++t) hist[bf16_exponent(x[t * tok_stride + h * ORC_D + c])] += 1;
            base3[h * ORC_D + c] = (uint8_t)best_window(hist, 8);
            base4[h * ORC_D + c] = (uint8_t)best_window(hist, 16);
        }
    }
}

/* ---- code plane location of code bit `bit` (0..2) of element s (format v3, as v1).
 * Unit u = s/32 owns words W0(u), W1(u), W2(u), word Wk(u) stored at byte
 * offset 8192 + 4*(k*256 + u).  Within the unit, j = s%32, half h = j/16,
 * jj = j%16, byte lane L = jj%4, quad q = jj/4:
 *   q=0: code bits 0..2 -> Wh, lane L, bits 0..2
 *   q=1: code bits 0..2 -> Wh, lane L, bits 3..5
 *   q=2: code bits 0..2 -> W2, lane L, bits 3h..3h+2
 *   q=3: code bits 0..1 -> Wh, lane L, bits 6..7; code bit 2 -> W2, lane L, bit 6+h
 * Returns the byte offset inside the slot image; *bitpos is the bit inside it. */
static int plane_bit_location(int plane, int s, int bit, int* bitpos) {
    int u = s / 32, j = s % 32, h = j / 16, jj = j % 16, lane = jj % 4, q = jj / 4;
    int word, pos;
    if (q == 0) { word = h; pos = bit; }
    else if (q == 1) { word = h; pos = 3 + bit; }
    else if (q == 2) { word = 2; pos = 3 * h + bit; }
    else if (bit < 2) { word = h; pos = 6 + bit; }
    else { word = 2; pos = 6 + h; }
    *bitpos = pos;
    return plane + 4 * (word * ORC_UNITS + u) + lane;
}
static int code_bit_location(int s, int bit, int* bitpos) { return plane_bit_location(ORC_OFF_CODE, s, bit, bitpos); }

/* A 3-bit field per element at plane offset `plane`, laid out like the code plane. */
static void put_field3(uint8_t* img, int plane, int s, unsigned v) {
    for (int b = 0; b < 3; ++b) {
        int pos;
        int at = plane_bit_location(plane, s, b, &pos);
        if ((v >> b) & 1u) img[at] |= (uint8_t)(1u << pos);
    }
}
static unsigned get_field3(const uint8_t* img, int plane, int s) {
    unsigned v = 0;
    for (int b = 0; b < 3; ++b) {
        int pos;
        int at = plane_bit_location(plane, s, b, &pos);
        v |= ((img[at] >> pos) & 1u) << b;
    }
    return v;
}

static void put_code(uint8_t* img, int s, unsigned code) {
    for (int b = 0; b < 3; ++b) {
        int pos;
        int at = code_bit_location(s, b, &pos);
        if ((code >> b) & 1u) img[at] |= (uint8_t)(1u << pos);
    }
}

static unsigned get_code(const uint8_t* img, int s) {
    unsigned code = 0;
    for (int b = 0; b < 3; ++b) {
        int pos;
        int at = code_bit_location(s, b, &pos);
        code |= ((img[at] >> pos) & 1u) << b;
    }
    return code;
}

/* ---- tag plane: group G's 2-bit mode at byte 11264 + G/4, bits 2*(G%4). */
static void put_tag(uint8_t* img, int G, unsigned mode) {
    img[ORC_OFF_TAG + G / 4] |= (uint8_t)((mode & 3u) << (2 * (G % 4)));
}
static unsigned get_tag(const uint8_t* img, int G) { return (img[ORC_OFF_TAG + G / 4] >> (2 * (G % 4))) & 3u; }

/* ---- mode rule (section 3.1): 3-bit if every offset from base3 is in [0,7],
 * else 4-bit if every offset from base4 is in [0,15], else raw.  Only the
 * elements with present[j] set count (present NULL: all eight). */
static unsigned choose_mode(const unsigned* e, const unsigned* b3, const unsigned* b4, const uint8_t* present) {
    int fits3 = 1, fits4 = 1;
    for (int j = 0; j < 8; ++j) {
        if (present && !present[j]) continue;
        int o3 = (int)e[j] - (int)b3[j];
        int o4 = (int)e[j] - (int)b4[j];
        if (o3 < 0 || o3 > 7) fits3 = 0;
        if (o4 < 0 || o4 > 15) fits4 = 0;
    }
    return fits3 ? ORC_M3BIT : (fits4 ? ORC_M4BIT : ORC_MRAW);
}

static int escape_bytes_of_mode(unsigned mode) { return mode == ORC_M3BIT ? 0 : (mode == ORC_M4BIT ? 1 : 8); }
int gaac_ref_escape_bytes_of_mode(int mode) { return escape_bytes_of_mode((unsigned)mode); }

/*
 * Encode the first n_tok tokens of a tile (1 <= n_tok <= 64; 64 = a full,
 * sealed tile).  `tile` is the tile in logical order [64 tokens][128
 * channels]; b3/b4 are the 128 per-channel bases of this (kv-head, K|V).
 * `forced` (NULL or 1024 modes) overrides the mode rule, for tests only.
 * `img` receives the slot image; it must hold 11536 + img_esc_cap bytes.
 * Returns the escape length in bytes (escape bytes only, the directory not
 * counted), or -1 if it exceeds img_esc_cap (the image is then incomplete).
 * Unused escape bytes stay zero.
 *
 * Codes: 3-bit group: e - base3; 4-bit group: (e - base4) & 7, with bit 3 of
 * element j's offset in bit j of the group's escape byte; raw group: code 0,
 * the eight exponents as eight escape bytes in element order.
 *
 * Open tiles (n_tok < 64; section 3.3 keeps the last block open while decode
 * tokens arrive, and the open block may be kept in its slot as it fills).  An element of
 * a token >= n_tok is absent: it takes no part in its group's mode (a group
 * with no present element is 3-bit), and every field it owns is zero: its
 * mantissa bits, the sign bit it lends to its neighbour's byte, its code, its
 * escape bit and, in a raw group, its exponent byte.  With every token present
 * this is the full tile's encoding, so a tile filled token by token ends in
 * the bytes of the tile encoded at once.
 */
static int encode_prefix(const uint16_t* tile, int n_tok, int kind, const uint8_t* base3, const uint8_t* base4,
                         const uint8_t* forced, uint8_t* img, int img_esc_cap) {
    memset(img, 0, (size_t)(ORC_OFF_ESC + img_esc_cap));
    uint16_t seq[ORC_TILE];
    uint8_t present[ORC_TILE];
    for (int t = 0; t < ORC_BLOCK; ++t)
        for (int c = 0; c < ORC_D; ++c) {
            int s = gaac_ref_storage_index(kind, t, c);
            present[s] = t < n_tok;
            seq[s] = present[s] ? tile[t * ORC_D + c] : 0;  /* absent: no sign, mantissa or exponent */
        }

    for (int s = 0; s < ORC_TILE; ++s)
        img[s] = (uint8_t)((bf16_signmant(seq[s]) & 0x7Fu) | (bf16_signmant(seq[sign_source(s)]) & 0x80u));

    /* pass 1: every group's mode over its present elements; the raw bytes follow all 4-bit bytes */
    unsigned modes[ORC_GROUPS];
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned e[8], b3[8], b4[8];
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            b3[j] = base3[channel_of(kind, s)];
            b4[j] = base4[channel_of(kind, s)];
            e[j] = bf16_exponent(seq[s]);
        }
        modes[G] = forced ? forced[G] : choose_mode(e, b3, b4, present + 8 * G);
        if (modes[G] == ORC_M4BIT) n4 += 1;
        if (modes[G] == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > img_esc_cap) return -1;

    /* pass 2: tags, codes, escape bytes, directory */
    int at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = modes[G];
        put_tag(img, G, mode);
        uint8_t esc4 = 0;
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            unsigned e = bf16_exponent(seq[s]), code = 0;
            if (!present[s]) {
                /* absent: code, escape bit and raw exponent byte stay zero */
            } else if (mode == ORC_M3BIT) {
                code = (e - base3[channel_of(kind, s)]) & 7u;
            } else if (mode == ORC_M4BIT) {
                unsigned off = (e - base4[channel_of(kind, s)]) & 0xFFu;
                code = off & 7u;
                esc4 |= (uint8_t)(((off >> 3) & 1u) << j);
            } else {
                img[ORC_OFF_ESC + n4 + 8 * atraw + j] = (uint8_t)e;
            }
            put_code(img, s, code);
        }
        if (mode == ORC_M4BIT) img[ORC_OFF_ESC + at4++] = esc4;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {  /* directory entry: groups so far */
            int w = G / ORC_DIR_GROUPS;
            unsigned entry = ((unsigned)at4 & 0x1FFu) | (((unsigned)atraw & 0x7Fu) << 9);
            img[ORC_OFF_DIR + 2 * w] = (uint8_t)(entry & 0xFFu);
            img[ORC_OFF_DIR + 2 * w + 1] = (uint8_t)(entry >> 8);
        }
    }
    return esc;
}

int gaac_ref_encode_tile(const uint16_t* tile, int kind, const uint8_t* base3, const uint8_t* base4,
                         const uint8_t* forced, uint8_t* img, int img_esc_cap) {
    return encode_prefix(tile, ORC_BLOCK, kind, base3, base4, forced, img, img_esc_cap);
}

int gaac_ref_encode_open_tile(const uint16_t* tile, int n_tok, int kind, const uint8_t* base3,
                              const uint8_t* base4, uint8_t* img, int img_esc_cap) {
    if (n_tok < 1 || n_tok > ORC_BLOCK) return -2;
    return encode_prefix(tile, n_tok, kind, base3, base4, NULL, img, img_esc_cap);
}

/*
 * Decode one slot image into the logical tile [64][128].
 * Returns the number of escape bytes the image uses, or -1 on a reserved tag
 * (3), -2 if the escape stream would run past esc_limit bytes, or -3 if a
 * directory entry differs from the group counts of the eighths it covers.
 */
int gaac_ref_decode_tile(const uint8_t* img, int kind, const uint8_t* base3, const uint8_t* base4,
                         int esc_limit, uint16_t* tile) {
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = get_tag(img, G);
        if (mode == 3u) return -1;
        if (mode == ORC_M4BIT) n4 += 1;
        if (mode == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > esc_limit) return -2;
    int at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = get_tag(img, G);
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            int c = channel_of(kind, s);
            unsigned code = get_code(img, s), e;
            if (mode == ORC_M3BIT) {
                e = base3[c] + code;
            } else if (mode == ORC_M4BIT) {
                e = base4[c] + (code | (((img[ORC_OFF_ESC + at4] >> j) & 1u) << 3));
            } else {
                e = img[ORC_OFF_ESC + n4 + 8 * atraw + j];
            }
            int t, cc;
            storage_to_tc(kind, s, &t, &cc);
            unsigned sm = (img[s] & 0x7Fu) | (img[sign_holder(s)] & 0x80u);
            tile[t * ORC_D + cc] = bf16_join(sm, e);
        }
        if (mode == ORC_M4BIT) at4 += 1;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {
            int w = G / ORC_DIR_GROUPS;
            int dir = img[ORC_OFF_DIR + 2 * w] | (img[ORC_OFF_DIR + 2 * w + 1] << 8);
            if (dir != ((at4 & 0x1FF) | ((atraw & 0x7F) << 9))) return -3;
        }
    }
    return esc;
}

/* Per-mode group counts of an encoded tile (diagnostics of section 4.7.1). */
void gaac_ref_mode_counts(const uint8_t* img, int64_t* counts4) {
    for (int m = 0; m < 4; ++m) counts4[m] = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) counts4[get_tag(img, G)] += 1;
}

/* Raw fallback image (section 3.3): the BF16 words in storage order. */
void gaac_ref_raw_tile(const uint16_t* tile, int kind, uint16_t* raw) {
    for (int t = 0; t < ORC_BLOCK; ++t)
        for (int c = 0; c < ORC_D; ++c) raw[gaac_ref_storage_index(kind, t, c)] = tile[t * ORC_D + c];
}
void gaac_ref_unraw_tile(const uint16_t* raw, int kind, uint16_t* tile) {
    for (int t = 0; t < ORC_BLOCK; ++t)
        for (int c = 0; c < ORC_D; ++c) tile[t * ORC_D + c] = raw[gaac_ref_storage_index(kind, t, c)];
}

/* ======================================================================
 * FP8 variant (GAAC page, Appendix B "Relation to FP8 KV": the same exponent
 * coding applied to an FP8 cache, E4M3 and E5M2).  The page prints only the
 * resulting ratios; this file fixes "GAAC-FP8 tile format v1":
 *   element     E4M3: sign(1) exponent(4) mantissa(3); E5M2: sign(1)
 *               exponent(5) mantissa(2); sm = sign << MW | mantissa
 *   tile, order, groups, modes, codes, tags, directory and escape area as in
 *               format v3, with the exponent windows inside the format's
 *               2^EW exponent values (E4M3 has one 16-window, base4 = 0, so
 *               it never needs the raw mode)
 *   slot image  E4M3: [0,4096) sm nibbles (element s in byte s/2, low nibble
 *                     for even s); [4096,7168) codes; [7168,7424) tags;
 *                     [7424,7440) directory; [7440,7936) escape area
 *               E5M2: [0,3072) sm, 3 bits per element laid out like the code
 *                     plane; [3072,6144) codes; [6144,6400) tags;
 *                     [6400,6416) directory; [6416,6912) escape area
 * ====================================================================== */
enum { ORC_FP8_E4M3 = 0, ORC_FP8_E5M2 = 1 };

typedef struct { int ew, mw, off_code, off_tag, off_dir, off_esc, slot; } fp8_layout;

static int fp8_layout_of(int fmt, fp8_layout* L) {
    if (fmt == ORC_FP8_E4M3) { fp8_layout l = {4, 3, 4096, 7168, 7424, 7440, 7936}; *L = l; return 1; }
    if (fmt == ORC_FP8_E5M2) { fp8_layout l = {5, 2, 3072, 6144, 6400, 6416, 6912}; *L = l; return 1; }
    return 0;
}

int gaac_ref_fp8_slot_bytes(int fmt) { fp8_layout L; return fp8_layout_of(fmt, &L) ? L.slot : 0; }

/* Windows of 8 and 16 exponents among the format's 2^EW values, from
 * x[t*tok_stride + h*128 + c] (FP8 bytes); ties go to the smallest base. */
int gaac_ref_fp8_calibrate(const uint8_t* x, int64_t n_tok, int64_t tok_stride, int n_heads, int fmt,
                           uint8_t* base3, uint8_t* base4) {
    fp8_layout L;
    if (!fp8_layout_of(fmt, &L)) return -1;
    int nb = 1 << L.ew;
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < ORC_D; ++c) {
            uint64_t hist[32];
            memset(hist, 0, sizeof hist);
            for (int64_t t = 0; t < n_tok; ++t) hist[(x[t * tok_stride + h * ORC_D + c] >> L.mw) & (nb - 1)] += 1;
            base3[h * ORC_D + c] = (uint8_t)best_window_n(hist, nb, 8);
            base4[h * ORC_D + c] = (uint8_t)best_window_n(hist, nb, 16);
        }
    }
    return 0;
}

static void fp8_put_sm(uint8_t* img, const fp8_layout* L, int s, unsigned sm) {
    if (L->ew == 4) img[s / 2] |= (uint8_t)((sm & 15u) << (4 * (s % 2)));
    else put_field3(img, 0, s, sm);
}
static unsigned fp8_get_sm(const uint8_t* img, const fp8_layout* L, int s) {
    if (L->ew == 4) return (img[s / 2] >> (4 * (s % 2))) & 15u;
    return get_field3(img, 0, s);
}

/* Encode one FP8 tile ([64][128] logical order); img must hold
 * off_esc + img_esc_cap bytes.  Returns the escape length or -1 past
 * img_esc_cap; -2 on a bad fmt. */
int gaac_ref_fp8_encode_tile(const uint8_t* tile, int kind, int fmt, const uint8_t* base3, const uint8_t* base4,
                             const uint8_t* forced, uint8_t* img, int img_esc_cap) {
    fp8_layout L;
    if (!fp8_layout_of(fmt, &L)) return -2;
    memset(img, 0, (size_t)(L.off_esc + img_esc_cap));
    uint8_t seq[ORC_TILE];
    for (int t = 0; t < ORC_BLOCK; ++t)
        for (int c = 0; c < ORC_D; ++c) seq[gaac_ref_storage_index(kind, t, c)] = tile[t * ORC_D + c];
    unsigned emask = (1u << L.ew) - 1u, mmask = (1u << L.mw) - 1u;
    for (int s = 0; s < ORC_TILE; ++s) fp8_put_sm(img, &L, s, ((seq[s] >> 7) << L.mw) | (seq[s] & mmask));
    unsigned modes[ORC_GROUPS];
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned e[8], b3[8], b4[8];
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            e[j] = (seq[s] >> L.mw) & emask;
            b3[j] = base3[channel_of(kind, s)];
            b4[j] = base4[channel_of(kind, s)];
        }
        modes[G] = forced ? forced[G] : choose_mode(e, b3, b4, NULL);
        if (modes[G] == ORC_M4BIT) n4 += 1;
        if (modes[G] == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > img_esc_cap) return -1;
    int at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = modes[G];
        img[L.off_tag + G / 4] |= (uint8_t)((mode & 3u) << (2 * (G % 4)));
        uint8_t esc4 = 0;
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            unsigned e = (seq[s] >> L.mw) & emask, code = 0;
            if (mode == ORC_M3BIT) {
                code = (e - base3[channel_of(kind, s)]) & 7u;
            } else if (mode == ORC_M4BIT) {
                unsigned off = (e - base4[channel_of(kind, s)]) & 0xFFu;
                code = off & 7u;
                esc4 |= (uint8_t)(((off >> 3) & 1u) << j);
            } else {
                img[L.off_esc + n4 + 8 * atraw + j] = (uint8_t)e;
            }
            put_field3(img, L.off_code, s, code);
        }
        if (mode == ORC_M4BIT) img[L.off_esc + at4++] = esc4;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {
            int w = G / ORC_DIR_GROUPS;
            unsigned entry = ((unsigned)at4 & 0x1FFu) | (((unsigned)atraw & 0x7Fu) << 9);
            img[L.off_dir + 2 * w] = (uint8_t)(entry & 0xFFu);
            img[L.off_dir + 2 * w + 1] = (uint8_t)(entry >> 8);
        }
    }
    return esc;
}

/* Decode one FP8 slot image into [64][128].  Returns the escape bytes used,
 * -1 on a reserved tag, -2 past esc_limit, -3 on a directory mismatch, -4 on
 * a bad fmt. */
int gaac_ref_fp8_decode_tile(const uint8_t* img, int kind, int fmt, const uint8_t* base3, const uint8_t* base4,
                             int esc_limit, uint8_t* tile) {
    fp8_layout L;
    if (!fp8_layout_of(fmt, &L)) return -4;
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = (img[L.off_tag + G / 4] >> (2 * (G % 4))) & 3u;
        if (mode == 3u) return -1;
        if (mode == ORC_M4BIT) n4 += 1;
        if (mode == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > esc_limit) return -2;
    unsigned emask = (1u << L.ew) - 1u;
    int at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = (img[L.off_tag + G / 4] >> (2 * (G % 4))) & 3u;
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j;
            int c = channel_of(kind, s);
            unsigned code = get_field3(img, L.off_code, s), e;
            if (mode == ORC_M3BIT) e = base3[c] + code;
            else if (mode == ORC_M4BIT) e = base4[c] + (code | (((img[L.off_esc + at4] >> j) & 1u) << 3));
            else e = img[L.off_esc + n4 + 8 * atraw + j];
            unsigned sm = fp8_get_sm(img, &L, s);
            int t, cc;
            storage_to_tc(kind, s, &t, &cc);
            tile[t * ORC_D + cc] = (uint8_t)(((sm >> L.mw) << 7) | ((e & emask) << L.mw) | (sm & ((1u << L.mw) - 1u)));
        }
        if (mode == ORC_M4BIT) at4 += 1;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {
            int w = G / ORC_DIR_GROUPS;
            int dir = img[L.off_dir + 2 * w] | (img[L.off_dir + 2 * w + 1] << 8);
            if (dir != ((at4 & 0x1FF) | ((atraw & 0x7F) << 9))) return -3;
        }
    }
    return esc;
}

void gaac_ref_fp8_mode_counts(const uint8_t* img, int fmt, int64_t* counts4) {
    fp8_layout L;
    for (int m = 0; m < 4; ++m) counts4[m] = 0;
    if (!fp8_layout_of(fmt, &L)) return;
    for (int G = 0; G < ORC_GROUPS; ++G) counts4[(img[L.off_tag + G / 4] >> (2 * (G % 4))) & 3u] += 1;
}

/* ---- decode attention in fp64 (section 3.2; grouped-query heads share a
 * kv-head, q head h reads kv-head h / (Hq/Hkv)).
 * q[hq*d + c]; k, v: element (t, hk, c) at t*tok_stride + hk*d + c; d = 128, or 256
 * for a head the storage splits into two 128-channel half-heads (Appendix D:
 * a 256-dimensional head is represented as two 128-dimensional half-heads; the
 * attention still runs over the whole head).
 * out[hq*128 + c] = sum_t softmax_t(scale * q.k_t) v_t[c]; T == 0 gives zeros.
 * flags (may be NULL), per q head, mark rows whose quantities leave the fp32
 * range, so that no fp32 evaluation of them can be held to a tolerance:
 *   bit 0: for some token, |scale| * sum_c |q_c k_tc| exceeds the largest
 *          finite fp32 value.  That sum bounds the logit scale * q.k_t and
 *          every partial sum of its terms scale * q_c * k_tc, so below it the
 *          logit has an fp32 value reachable in any order of summation.
 *   bit 1: for some channel, sum_t w_t |v_tc| exceeds the largest finite fp32
 *          value, w_t = exp(logit_t - max logit) being the unnormalised
 *          softmax weight (at most 1): the numerator of the softmax-weighted
 *          sum then has no fp32 value.
 * Such rows are reported apart from the ones compared with a tolerance. */
static double bf16_to_double(uint16_t x) {
    uint32_t u = (uint32_t)x << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void gaac_ref_attention_d(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t tok_stride, int64_t T,
                          int Hq, int Hkv, int d, double scale, double* out, int32_t* flags, double* logits_scratch) {
    int r = Hq / Hkv;
    for (int hq = 0; hq < Hq; ++hq) {
        int hk = hq / r;
        int32_t flag = 0;
        for (int c = 0; c < d; ++c) out[hq * d + c] = 0.0;
        if (T == 0) { if (flags) flags[hq] = 0; continue; }
        double m = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            double dot = 0.0, mag = 0.0;
            for (int c = 0; c < d; ++c) {
                double qc = bf16_to_double(q[hq * d + c]);
                double kc = bf16_to_double(k[t * tok_stride + hk * d + c]);
                dot += qc * kc;
                mag += fabs(qc * kc);
            }
            if (fabs(scale) * mag > 3.4028234663852886e38) flag |= 1;
            logits_scratch[t] = scale * dot;
            if (logits_scratch[t] > m) m = logits_scratch[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double w = exp(logits_scratch[t] - m);
            logits_scratch[t] = w;
            l += w;
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0, mag = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                double vc = bf16_to_double(v[t * tok_stride + hk * d + c]);
                acc += logits_scratch[t] * vc;
                mag += logits_scratch[t] * fabs(vc);
            }
            if (mag > 3.4028234663852886e38) flag |= 2;
            out[hq * d + c] = acc / l;
        }
        if (flags) flags[hq] = flag;
    }
}

void gaac_ref_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t tok_stride, int64_t T,
                        int Hq, int Hkv, double scale, double* out, int32_t* flags, double* logits_scratch) {
    gaac_ref_attention_d(q, k, v, tok_stride, T, Hq, Hkv, ORC_D, scale, out, flags, logits_scratch);
}

/* ==== Nested 2-bit mode: the ablation format of section 4.7.2 (Table 4) ====
 *
 * The page measures a fourth, 2-bit mode nested inside the 3-bit one: a group
 * whose offsets from a per-channel base2 all fit [0,3] keeps 2 code bits per
 * element.  The saving only exists if the code width varies per group, so this
 * ablation format (not used by the cache) replaces format v3's fixed 3-bit
 * code planes with a code stream:
 *   [0,8192)       sign|mantissa plane, as format v3
 *   [8192,11264)   code stream: groups in group order; a 2-bit group takes 16
 *                  bits, a 3-bit or 4-bit group 24 (the 4-bit group's low
 *                  three offset bits), a raw group none; element j of a group
 *                  at bit (group start + j * width); bit b of the stream is bit
 *                  b % 8 of byte b / 8; zero past its end
 *   [11264,11520)  tags, 2 bits per group: 0 3-bit, 1 4-bit, 2 raw, 3 2-bit
 *   [11520,11552)  directory: 8 u32, entry w = 4-bit groups | raw groups << 9
 *                  | code-stream bits << 16, each over groups [0, 128(w+1))
 *   [11552,12048)  escape area, capacity 496: one byte per 4-bit group, then
 *                  eight exponent bytes per raw group, each in group order
 * The mode rule tries the windows from the narrowest: 2-bit if every offset
 * from base2 is in [0,3], else 3-bit, else 4-bit, else raw.
 */
#define NST_OFF_CODE 8192
#define NST_OFF_TAG 11264
#define NST_OFF_DIR 11520
#define NST_OFF_ESC 11552
#define NST_SLOT (NST_OFF_ESC + ORC_ESC_CAP)
enum { NST_M2BIT = 3 };

int gaac_ref_nested_slot_bytes(void) { return NST_SLOT; }

/* base2 of every (head, channel): the 4-exponent window holding the most
 * calibration values (ties to the smallest base), as base3 and base4. */
void gaac_ref_nested_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_heads, uint8_t* base2) {
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < ORC_D; ++c) {
            uint64_t hist[256];
            memset(hist, 0, sizeof hist);
            for (int64_t t = 0; t < n_tok; ++t) hist[bf16_exponent(x[t * tok_stride + h * ORC_D + c])] += 1;
            base2[h * ORC_D + c] = (uint8_t)best_window(hist, 4);
        }
    }
}

static int nested_width(unsigned mode) { return mode == NST_M2BIT ? 2 : (mode == ORC_MRAW ? 0 : 3); }

static void put_bits(uint8_t* img, int bit, unsigned v, int n) {
    for (int i = 0; i < n; ++i)
        if ((v >> i) & 1u) img[NST_OFF_CODE + (bit + i) / 8] |= (uint8_t)(1u << ((bit + i) % 8));
}
static unsigned get_bits(const uint8_t* img, int bit, int n) {
    unsigned v = 0;
    for (int i = 0; i < n; ++i) v |= ((img[NST_OFF_CODE + (bit + i) / 8] >> ((bit + i) % 8)) & 1u) << i;
    return v;
}

/* Encode one full tile ([64][128], logical order).  Returns the escape length,
 * or -1 if the escape stream exceeds 496 bytes; *code_bits receives the length
 * of the code stream in bits.  img must hold NST_SLOT bytes. */
int gaac_ref_nested_encode_tile(const uint16_t* tile, int kind, const uint8_t* base2, const uint8_t* base3,
                                const uint8_t* base4, uint8_t* img, int* code_bits) {
    memset(img, 0, NST_SLOT);
    uint16_t seq[ORC_TILE];
    for (int t = 0; t < ORC_BLOCK; ++t)
        for (int c = 0; c < ORC_D; ++c) seq[gaac_ref_storage_index(kind, t, c)] = tile[t * ORC_D + c];
    for (int s = 0; s < ORC_TILE; ++s)
        img[s] = (uint8_t)((bf16_signmant(seq[s]) & 0x7Fu) | (bf16_signmant(seq[sign_source(s)]) & 0x80u));
    unsigned modes[ORC_GROUPS];
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned e[8], b3[8], b4[8];
        int fits2 = 1;
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j, c = channel_of(kind, s);
            e[j] = bf16_exponent(seq[s]);
            b3[j] = base3[c];
            b4[j] = base4[c];
            int o2 = (int)e[j] - (int)base2[c];
            if (o2 < 0 || o2 > 3) fits2 = 0;
        }
        modes[G] = fits2 ? NST_M2BIT : choose_mode(e, b3, b4, NULL);
        if (modes[G] == ORC_M4BIT) n4 += 1;
        if (modes[G] == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > ORC_ESC_CAP) return -1;
    int bit = 0, at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = modes[G];
        int w = nested_width(mode);
        img[NST_OFF_TAG + G / 4] |= (uint8_t)(mode << (2 * (G % 4)));
        uint8_t esc4 = 0;
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j, c = channel_of(kind, s);
            unsigned e = bf16_exponent(seq[s]);
            if (mode == NST_M2BIT) {
                put_bits(img, bit + 2 * j, e - base2[c], 2);
            } else if (mode == ORC_M3BIT) {
                put_bits(img, bit + 3 * j, e - base3[c], 3);
            } else if (mode == ORC_M4BIT) {
                unsigned off = (e - base4[c]) & 0xFFu;
                put_bits(img, bit + 3 * j, off & 7u, 3);
                esc4 |= (uint8_t)(((off >> 3) & 1u) << j);
            } else {
                img[NST_OFF_ESC + n4 + 8 * atraw + j] = (uint8_t)e;
            }
        }
        bit += 8 * w;
        if (mode == ORC_M4BIT) img[NST_OFF_ESC + at4++] = esc4;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {
            uint32_t entry = ((uint32_t)at4 & 0x1FFu) | (((uint32_t)atraw & 0x7Fu) << 9) | ((uint32_t)bit << 16);
            memcpy(img + NST_OFF_DIR + 4 * (G / ORC_DIR_GROUPS), &entry, 4);  /* little-endian host assumed */
        }
    }
    if (code_bits) *code_bits = bit;
    return esc;
}

/* Decode a nested-format image into the logical tile.  Returns the escape
 * length, -2 if the escape stream exceeds 496 bytes, or -3 if a directory
 * entry differs from the counts of the groups it covers. */
int gaac_ref_nested_decode_tile(const uint8_t* img, int kind, const uint8_t* base2, const uint8_t* base3,
                                const uint8_t* base4, uint16_t* tile) {
    int n4 = 0, nraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = (img[NST_OFF_TAG + G / 4] >> (2 * (G % 4))) & 3u;
        if (mode == ORC_M4BIT) n4 += 1;
        if (mode == ORC_MRAW) nraw += 1;
    }
    int esc = n4 + 8 * nraw;
    if (esc > ORC_ESC_CAP) return -2;
    int bit = 0, at4 = 0, atraw = 0;
    for (int G = 0; G < ORC_GROUPS; ++G) {
        unsigned mode = (img[NST_OFF_TAG + G / 4] >> (2 * (G % 4))) & 3u;
        int w = nested_width(mode);
        for (int j = 0; j < 8; ++j) {
            int s = 8 * G + j, c = channel_of(kind, s);
            unsigned e;
            if (mode == NST_M2BIT) {
                e = base2[c] + get_bits(img, bit + 2 * j, 2);
            } else if (mode == ORC_M3BIT) {
                e = base3[c] + get_bits(img, bit + 3 * j, 3);
            } else if (mode == ORC_M4BIT) {
                e = base4[c] + (get_bits(img, bit + 3 * j, 3) | (((img[NST_OFF_ESC + at4] >> j) & 1u) << 3));
            } else {
                e = img[NST_OFF_ESC + n4 + 8 * atraw + j];
            }
            int t, cc;
            storage_to_tc(kind, s, &t, &cc);
            unsigned sm = (img[s] & 0x7Fu) | (img[sign_holder(s)] & 0x80u);
            tile[t * ORC_D + cc] = bf16_join(sm, e & 0xFFu);
        }
        bit += 8 * w;
        if (mode == ORC_M4BIT) at4 += 1;
        if (mode == ORC_MRAW) atraw += 1;
        if ((G + 1) % ORC_DIR_GROUPS == 0) {
            uint32_t entry;
            memcpy(&entry, img + NST_OFF_DIR + 4 * (G / ORC_DIR_GROUPS), 4);
            if (entry != (((uint32_t)at4 & 0x1FFu) | (((uint32_t)atraw & 0x7Fu) << 9) | ((uint32_t)bit << 16)))
                return -3;
        }
    }
    return esc;
}
