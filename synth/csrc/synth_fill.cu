// Device-side fill of arena slots with seeded synthetic MXFP4 experts.
//
// Input generation only (no part of the method): the same counter-based
// SplitMix64 streams as synth/__init__.py, so that any expert written here can
// be regenerated on the host byte for byte. Expert (layer, expert) is keyed by
// its flat id layer * E + expert.
//   codes byte j  = byte (j % 8) of hash(j / 8)            (uniform nibbles)
//   scale byte j  = 121 + ((hash(j / 32) >> 2 * (j % 32)) & 3)   (2^U, U in -6..-3)
// where j is the row-major index; codes are stored in tile-major 16 KB blocks
// and scales in tile-atom order (the arena record layout).
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t stream_base(uint64_t seed, uint32_t tid, uint32_t a, uint32_t b) {
    const uint64_t key = ((uint64_t)(tid & 0xFF) << 56) ^ ((uint64_t)(a & 0xFFFFFFF) << 28) ^ (uint64_t)(b & 0xFFFFFFF);
    return mix(seed ^ mix(key));
}

__device__ inline uint64_t hash_at(uint64_t base, uint64_t idx) { return mix(base + (idx + 1) * kGamma); }

struct Region {
    int64_t off;
    int64_t bytes;    // logical bytes (rows x bytes per row)
    uint32_t tid;
    int scales;       // codes: 0; scales: 1 (gate/up matrix) or 2 (down matrix)
    int kb;           // bytes per row: K / 2 for codes, K / 32 for scales
    int ffn;
    int gate_up;      // codes: 1 for the gate/up matrix
};

// Tile (128 consecutive rows) and tile row of a logical row.
__device__ inline void tile_of(int64_t row, int64_t* tile, int64_t* tr) {
    *tile = row / 128;
    *tr = row % 128;
}

// Position of logical code byte `col` of `row` in the tile-major block order:
// 16 KB blocks of 128 rows x 128 bytes per (tile, chunk of 128 bytes along the
// row), 16-byte piece c of tile row r at piece c ^ (r % 8).
__device__ inline int64_t packed_code_offset(const Region& r, int64_t row, int64_t col) {
    int64_t tile, tr;
    tile_of(row, &tile, &tr);
    const int64_t nkc = (r.kb + 127) / 128;
    const int64_t kc = col / 128, piece = (col % 128) / 16;
    return (tile * nkc + kc) * 16384 + tr * 128 + ((piece ^ (tr & 7)) * 16) + col % 16;
}

// Position of logical scale byte (row, k-block) in the arena's tile-atom order:
// 128-row tiles, 512-byte atoms of 4 k-blocks, byte (r % 32) * 16 + (r / 32) * 4 + kb % 4.
__device__ inline int64_t packed_scale_offset(const Region& r, int64_t row, int kb) {
    int64_t tile, tr;
    tile_of(row, &tile, &tr);
    const int64_t atoms_per_tile = r.kb / 4;
    return (tile * atoms_per_tile + kb / 4) * 512 + (tr % 32) * 16 + (tr / 32) * 4 + kb % 4;
}

__global__ void fill_slots(uint8_t* arena, int64_t slot_bytes, Region r0, Region r1, Region r2, Region r3,
                           const int32_t* slots, const int32_t* flats, int slot_begin, int n, int E, uint64_t seed) {
    const int item = blockIdx.y;
    if (item >= n) return;
    const int slot = slots ? slots[item] : slot_begin + item;
    const int flat = flats[slots ? item : slot];
    if (slot < 0 || flat < 0) return;
    const uint32_t layer = (uint32_t)(flat / E), expert = (uint32_t)(flat % E);
    uint8_t* rec = arena + (size_t)slot * slot_bytes;
    const Region rs[4] = {r0, r1, r2, r3};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const Region r = rs[q];
        const uint64_t base = stream_base(seed, r.tid, layer, expert);
        if (!r.scales) {
            const int64_t words = r.bytes / 8;              // 8 logical bytes stay within one 16-byte piece
            for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words; w += (int64_t)gridDim.x * blockDim.x) {
                const int64_t row = (w * 8) / r.kb, col = (w * 8) % r.kb;
                *reinterpret_cast<uint64_t*>(rec + r.off + packed_code_offset(r, row, col)) = hash_at(base, (uint64_t)w);
            }
        } else {
            uint8_t* dstb = rec + r.off;
            const int64_t groups = r.bytes / 32;                 // one hash -> 32 logical scale bytes
            for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += (int64_t)gridDim.x * blockDim.x) {
                const uint64_t h = hash_at(base, (uint64_t)g);
                for (int j = 0; j < 32; ++j) {
                    const int64_t idx = g * 32 + j;              // logical row-major index
                    const int64_t row = idx / r.kb;
                    const int kb = (int)(idx % r.kb);
                    dstb[packed_scale_offset(r, row, kb)] = (uint8_t)(121u + (uint32_t)((h >> (2 * j)) & 3u));
                }
            }
        }
    }
}

}  // namespace

extern "C" {

// Fill slots with seeded experts.
//   slots == NULL : slots [slot_begin, slot_begin + n), expert flats[slot] (flats = owner table, -1 skips)
//   slots != NULL : slot slots[i] gets expert flats[i], i < n
// All pointers are device pointers except the scalar arguments. Returns a cudaError_t value.
int synth_fill_slots(void* arena_base, int64_t slot_bytes, int64_t off_gu_codes, int64_t off_gu_scales,
                     int64_t off_dn_codes, int64_t off_dn_scales, int d, int ffn, const int32_t* slots,
                     const int32_t* flats, int slot_begin, int n, int E, uint64_t seed, void* stream) {
    if (n <= 0) return 0;
    Region r0{off_gu_codes, (int64_t)2 * ffn * d / 2, 4, 0, d / 2, ffn, 1};
    Region r1{off_gu_scales, (int64_t)2 * ffn * d / 32, 5, 1, d / 32, ffn, 0};
    Region r2{off_dn_codes, (int64_t)d * ffn / 2, 6, 0, ffn / 2, ffn, 0};
    Region r3{off_dn_scales, (int64_t)d * ffn / 32, 7, 2, ffn / 32, ffn, 0};
    dim3 grid(64, n);
    fill_slots<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t*>(arena_base), slot_bytes,
                                                                    r0, r1, r2, r3, slots, flats, slot_begin, n, E,
                                                                    seed);
    return (int)cudaGetLastError();
}

}  // extern "C"
