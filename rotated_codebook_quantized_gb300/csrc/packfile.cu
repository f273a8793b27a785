// Persisted packed format: quantized layers written once and loaded without
// repeating the encode, with the bit width of each layer recovered from the
// size of its stored codebook.
//
// "How it works", "The ternary tier (1.58 bits)": the format marks itself (a
// codebook of 2^b entries means bit-packed, 3 entries trit-packed), so a model
// can mix tiers layer by layer; "Configuration that converter and loader
// share": the bit width is recovered from the saved codebook's size, never
// trusted from a config field, and the rotation and seed are recorded.  The
// weight-reservoir page: a flat, page-aligned binary file (a blob of indices
// and one of scales per layer, a small header with shapes and the rotation
// seed), loaded byte-identical to what was written.
//
// Layout (all integers little-endian; host code, no GPU involved):
//   [0, 64)         file header: magic "TQPACK\0\1", version, layer count, table offset
//   [64, 64+256 n)  one 256-byte record per layer (name, shape, group, stride,
//                   rotation dim / block / seed, blob offsets and sizes)
//   then, for each layer, three blobs each starting on a 4096-byte boundary:
//                   the codebook (levels fp64 centroids, ascending), the code
//                   words [experts][rows][row_stride] uint32 and the fp16
//                   scales [experts][rows][cols/group]; zero bytes in between.
#include <stdio.h>
#include <string.h>

#include <vector>

#include "tq.h"

namespace {

constexpr char kMagic[8] = {'T', 'Q', 'P', 'A', 'C', 'K', 0, 1};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kPage = 4096;
constexpr uint64_t kHeaderBytes = 64;
constexpr uint64_t kRecordBytes = 256;

struct FileHeader {
    char magic[8];
    uint32_t version;
    uint32_t n_layers;
    uint64_t table_offset;
    uint64_t file_bytes;
    uint8_t reserved[32];
};
static_assert(sizeof(FileHeader) == kHeaderBytes, "header size");

struct LayerRecord {
    char name[TQ_LAYER_NAME_BYTES];
    int32_t experts, rows, cols, group;
    int64_t row_stride_words;
    int32_t rot_dim, rot_block;
    uint64_t rot_seed;
    uint64_t codebook_offset, codebook_bytes;
    uint64_t codes_offset, codes_bytes;
    uint64_t scales_offset, scales_bytes;
    uint8_t reserved[kRecordBytes - TQ_LAYER_NAME_BYTES - 4 * 4 - 8 - 2 * 4 - 8 - 6 * 8];
};
static_assert(sizeof(LayerRecord) == kRecordBytes, "record size");

uint64_t round_page(uint64_t v) { return (v + kPage - 1) / kPage * kPage; }

bool levels_ok(int levels) { return levels == 3 || levels == 4 || levels == 8 || levels == 16 || levels == 256; }

int codes_per_word(int levels) {
    switch (levels) {
        case 3: return 20;
        case 4: return 16;
        case 8: return 10;
        case 16: return 8;
        case 256: return 4;
        default: return 0;
    }
}

// Checks a layer description and returns its blob sizes.
tq_status layer_sizes(const tq_layer_desc_t& d, uint64_t& cb, uint64_t& codes, uint64_t& scales) {
    if (!levels_ok(d.levels) || d.experts <= 0 || d.rows <= 0 || d.cols <= 0) return TQ_ERR_INVALID;
    if (!(d.group == 16 || d.group == 32 || d.group == 64 || d.group == 128) || d.cols % d.group) return TQ_ERR_INVALID;
    const int64_t words = (d.cols + codes_per_word(d.levels) - 1) / codes_per_word(d.levels);
    if (d.row_stride_words < words) return TQ_ERR_INVALID;
    if (d.rot_block <= 0 || d.rot_dim != d.cols || d.cols % d.rot_block) return TQ_ERR_INVALID;
    if (memchr(d.name, 0, TQ_LAYER_NAME_BYTES) == nullptr) return TQ_ERR_INVALID;  // unterminated name
    cb = (uint64_t)d.levels * 8;
    codes = (uint64_t)d.experts * d.rows * d.row_stride_words * 4;
    scales = (uint64_t)d.experts * d.rows * (d.cols / d.group) * 2;
    return TQ_OK;
}

bool write_at(FILE* f, uint64_t off, const void* p, uint64_t n) {
    if (fseeko(f, (off_t)off, SEEK_SET) != 0) return false;
    return n == 0 || fwrite(p, 1, n, f) == n;
}

bool read_at(FILE* f, uint64_t off, void* p, uint64_t n) {
    if (fseeko(f, (off_t)off, SEEK_SET) != 0) return false;
    return n == 0 || fread(p, 1, n, f) == n;
}

// Reads and validates the header and the layer table.
tq_status read_table(FILE* f, FileHeader& h, std::vector<LayerRecord>& recs) {
    if (!read_at(f, 0, &h, sizeof h)) return TQ_ERR_INVALID;
    if (memcmp(h.magic, kMagic, 8) != 0 || h.version != kVersion || h.table_offset != kHeaderBytes)
        return TQ_ERR_INVALID;
    if (h.n_layers > (1u << 20)) return TQ_ERR_INVALID;
    if (fseeko(f, 0, SEEK_END) != 0 || (uint64_t)ftello(f) != h.file_bytes) return TQ_ERR_INVALID;  // truncated
    recs.resize(h.n_layers);
    if (h.n_layers && !read_at(f, h.table_offset, recs.data(), (uint64_t)h.n_layers * kRecordBytes))
        return TQ_ERR_INVALID;
    for (const LayerRecord& r : recs) {
        if (memchr(r.name, 0, TQ_LAYER_NAME_BYTES) == nullptr) return TQ_ERR_INVALID;
        if (r.codebook_bytes % 8 || !levels_ok((int)(r.codebook_bytes / 8))) return TQ_ERR_INVALID;
        const uint64_t ends[3] = {r.codebook_offset + r.codebook_bytes, r.codes_offset + r.codes_bytes,
                                  r.scales_offset + r.scales_bytes};
        for (uint64_t e : ends)
            if (e > h.file_bytes) return TQ_ERR_INVALID;
    }
    return TQ_OK;
}

void fill_info(const LayerRecord& r, tq_layer_desc_t& d) {
    memcpy(d.name, r.name, TQ_LAYER_NAME_BYTES);
    d.experts = r.experts;
    d.rows = r.rows;
    d.cols = r.cols;
    d.group = r.group;
    d.row_stride_words = r.row_stride_words;
    d.levels = (int32_t)(r.codebook_bytes / 8);  // the width comes from the stored codebook
    d.rot_dim = r.rot_dim;
    d.rot_block = r.rot_block;
    d.rot_seed = r.rot_seed;
}

}  // namespace

extern "C" tq_status tq_layer_tier(const char* name, const tq_tier_policy_t* policy, int32_t* levels, int32_t* group) {
    if (!name || !policy || !levels || !group) return TQ_ERR_INVALID;
    // the first class whose marker the name contains decides; down projections before experts, so
    // that an expert's down projection takes the down-projection tier
    if (strstr(name, "down_proj")) {
        *levels = policy->down_levels;
        *group = policy->down_group;
    } else if (strstr(name, "expert")) {
        *levels = policy->expert_levels;
        *group = policy->expert_group;
    } else if (strstr(name, "mlp")) {
        *levels = policy->mlp_levels;
        *group = policy->mlp_group;
    } else if (strstr(name, "attn")) {
        *levels = policy->attn_levels;
        *group = policy->attn_group;
    } else {
        *levels = policy->other_levels;
        *group = policy->other_group;
    }
    return levels_ok(*levels) && (*group == 16 || *group == 32 || *group == 64 || *group == 128) ? TQ_OK
                                                                                                : TQ_ERR_INVALID;
}

extern "C" tq_status tq_pack_file_write(const char* path, const tq_layer_desc_t* layers, int32_t n_layers) {
    if (!path || n_layers < 0 || (n_layers > 0 && !layers)) return TQ_ERR_INVALID;
    std::vector<LayerRecord> recs(n_layers);
    uint64_t off = round_page(kHeaderBytes + (uint64_t)n_layers * kRecordBytes);
    for (int i = 0; i < n_layers; ++i) {
        const tq_layer_desc_t& d = layers[i];
        uint64_t cb, codes, scales;
        const tq_status s = layer_sizes(d, cb, codes, scales);
        if (s != TQ_OK) return s;
        if (!d.centroids || !d.codes || !d.scales) return TQ_ERR_INVALID;
        LayerRecord& r = recs[i];
        memset(&r, 0, sizeof r);
        memcpy(r.name, d.name, strlen(d.name));  // bytes after the terminator stay zero
        r.experts = d.experts;
        r.rows = d.rows;
        r.cols = d.cols;
        r.group = d.group;
        r.row_stride_words = d.row_stride_words;
        r.rot_dim = d.rot_dim;
        r.rot_block = d.rot_block;
        r.rot_seed = d.rot_seed;
        r.codebook_offset = off;
        r.codebook_bytes = cb;
        off = round_page(off + cb);
        r.codes_offset = off;
        r.codes_bytes = codes;
        off = round_page(off + codes);
        r.scales_offset = off;
        r.scales_bytes = scales;
        off = round_page(off + scales);
    }
    FileHeader h;
    memset(&h, 0, sizeof h);
    memcpy(h.magic, kMagic, 8);
    h.version = kVersion;
    h.n_layers = (uint32_t)n_layers;
    h.table_offset = kHeaderBytes;
    h.file_bytes = off;
    FILE* f = fopen(path, "wb");
    if (!f) return TQ_ERR_INVALID;
    bool ok = write_at(f, 0, &h, sizeof h) &&
              (n_layers == 0 || write_at(f, kHeaderBytes, recs.data(), (uint64_t)n_layers * kRecordBytes));
    for (int i = 0; i < n_layers && ok; ++i) {
        const LayerRecord& r = recs[i];
        ok = write_at(f, r.codebook_offset, layers[i].centroids, r.codebook_bytes) &&
             write_at(f, r.codes_offset, layers[i].codes, r.codes_bytes) &&
             write_at(f, r.scales_offset, layers[i].scales, r.scales_bytes);
    }
    // the padding after the last blob is part of the file: write its last byte explicitly
    if (ok && off > 0) {
        const uint8_t z = 0;
        uint64_t last = 0;
        if (n_layers > 0) last = recs[n_layers - 1].scales_offset + recs[n_layers - 1].scales_bytes;
        else last = kHeaderBytes;
        if (last < off) ok = write_at(f, off - 1, &z, 1);
    }
    if (fclose(f) != 0) ok = false;
    return ok ? TQ_OK : TQ_ERR_INVALID;
}

extern "C" tq_status tq_pack_file_info(const char* path, int32_t* n_layers, tq_layer_desc_t* infos, int32_t cap) {
    if (!path || !n_layers || cap < 0 || (cap > 0 && !infos)) return TQ_ERR_INVALID;
    FILE* f = fopen(path, "rb");
    if (!f) return TQ_ERR_INVALID;
    FileHeader h;
    std::vector<LayerRecord> recs;
    const tq_status s = read_table(f, h, recs);
    fclose(f);
    if (s != TQ_OK) return s;
    *n_layers = (int32_t)h.n_layers;
    for (int i = 0; i < (int)h.n_layers && i < cap; ++i) {
        memset(&infos[i], 0, sizeof infos[i]);
        fill_info(recs[i], infos[i]);
    }
    return TQ_OK;
}

extern "C" tq_status tq_pack_file_read_layer(const char* path, int32_t index, double* centroids, uint32_t* codes,
                                             uint16_t* scales) {
    if (!path || index < 0 || !centroids || !codes || !scales) return TQ_ERR_INVALID;
    FILE* f = fopen(path, "rb");
    if (!f) return TQ_ERR_INVALID;
    FileHeader h;
    std::vector<LayerRecord> recs;
    tq_status s = read_table(f, h, recs);
    if (s == TQ_OK && index >= (int)h.n_layers) s = TQ_ERR_INVALID;
    if (s == TQ_OK) {
        const LayerRecord& r = recs[index];
        if (!read_at(f, r.codebook_offset, centroids, r.codebook_bytes) ||
            !read_at(f, r.codes_offset, codes, r.codes_bytes) || !read_at(f, r.scales_offset, scales, r.scales_bytes))
            s = TQ_ERR_INVALID;
    }
    fclose(f);
    return s;
}
