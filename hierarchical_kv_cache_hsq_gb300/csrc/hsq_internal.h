// Internal declarations shared by the host (hsq_host.cpp) and device
// (hsq_kernels.cu) translation units of the HSQ library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "hsq.h"

namespace hsq {

constexpr int kDim = 128;
constexpr int kRopeLoRows = 256;            // positions p & 255
constexpr int kRopeRowFloats = kDim;        // cos[64] | sin[64]
constexpr int kCodebookFloats = 48;         // c4[16] | t4[15] pad | c3[8] | t3[7] pad
constexpr int kGsumFloats = 2 * 128 + 4;    // growth sums: RoPE'd keys | values | count | pad
constexpr int kPartStride = 132;            // acc[128] | m | l | pad | pad
constexpr int kMaxHotSlots = 1024;          // largest hot-group table per (b, KV head)

inline int groups_of(int T, int N) { return (T + N - 1) / N; }
inline int bitmap_words(int T) { return (T + 31) / 32; }
inline size_t record_bytes(int N) { return (size_t)N * 136; }

// float64 Lloyd-Max codebook for one coordinate of a uniform unit vector in R^dim.
bool lloyd_max(int bits, int dim, double* centroids, double* boundaries);

// Codebook block for the device: c4[16], t4[15] (+1 pad), c3[8], t3[7] (+1 pad).
void device_codebook(float out[kCodebookFloats]);

// RoPE angle tables: hi[a] = cos/sin(256 a omega_i), lo[c] = cos/sin(c omega_i), float64 -> float32.
void rope_tables(double theta, int max_pos, std::vector<float>& hi, std::vector<float>& lo);

// Configuration / cache validation; returns an empty string when valid.
std::string check_config(const hsq_config* cfg);
std::string check_cache_shape(const hsq_config* cfg, const hsq_cache* c);

// Process-wide fault-injection mask and last process-level error.
unsigned fault_mask();
void set_process_error(const std::string& s);
const char* process_error();

}  // namespace hsq
