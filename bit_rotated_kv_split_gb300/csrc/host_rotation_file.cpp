// Rotation file: a model's fixed per-layer rotations and clip thresholds on
// disk, written once after the offline calibration and read back at serving
// start-up.  myzaker.com OSCAR article, closing part (the code release ships
// a zoo of precomputed fixed rotations per model); gist.science "OSCAR:
// Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", Technical summary 2.2 A (R and the clip thresholds are
// computed once, offline, per layer).
//
// Layout (little-endian, this library's format):
//   bytes 0..7    magic "OSCARROT"
//   u32           version (1)
//   u32           n_layers L, u32 n_kv_heads H, u32 head_dim d
//   per layer l:  f32 tau_k, f32 tau_v, R_K [H][d][d] f32, R_V [H][d][d] f32
//   u64           FNV-1a (64-bit) of every byte before it
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "oscar.h"
#include "trace.h"

namespace {

constexpr char kMagic[8] = {'O', 'S', 'C', 'A', 'R', 'R', 'O', 'T'};
constexpr uint32_t kVersion = 1;

struct Fnv1a {
  uint64_t h = 1469598103934665603ull;
  void add(const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    for (size_t i = 0; i < n; ++i) {
      h ^= b[i];
      h *= 1099511628211ull;
    }
  }
};

bool little_endian() {
  const uint32_t one = 1;
  unsigned char c;
  std::memcpy(&c, &one, 1);
  return c == 1;
}

bool dims_ok(int32_t n_layers, int32_t n_kv_heads, int32_t d) {
  return n_layers >= 1 && n_kv_heads >= 1 && d >= 1 && d <= 1024 && int64_t(n_layers) * n_kv_heads <= (1 << 20);
}

struct File {
  std::FILE* f = nullptr;
  ~File() {
    if (f) std::fclose(f);
  }
};

}  // namespace

extern "C" oscar_status oscar_rotation_file_write(const char* path, int32_t n_layers, int32_t n_kv_heads, int32_t d,
                                                   const float* r_k, const float* r_v, const float* tau_k,
                                                   const float* tau_v) {
  OSCAR_TRACE_CALL();
  if (!path || !r_k || !r_v || !tau_k || !tau_v || !dims_ok(n_layers, n_kv_heads, d)) return OSCAR_ERR_INVALID_ARG;
  if (!little_endian()) return OSCAR_ERR_UNSUPPORTED;
  File out;
  out.f = std::fopen(path, "wb");
  if (!out.f) return OSCAR_ERR_FILE;
  Fnv1a sum;
  auto put = [&](const void* p, size_t n) {
    sum.add(p, n);
    return std::fwrite(p, 1, n, out.f) == n;
  };
  const uint32_t head[4] = {kVersion, uint32_t(n_layers), uint32_t(n_kv_heads), uint32_t(d)};
  bool ok = put(kMagic, sizeof(kMagic)) && put(head, sizeof(head));
  const size_t per = size_t(n_kv_heads) * d * d;
  for (int32_t l = 0; ok && l < n_layers; ++l) {
    ok = put(tau_k + l, 4) && put(tau_v + l, 4) && put(r_k + l * per, per * 4) && put(r_v + l * per, per * 4);
  }
  const uint64_t h = sum.h;
  ok = ok && std::fwrite(&h, 1, 8, out.f) == 8;
  ok = std::fclose(out.f) == 0 && ok;
  out.f = nullptr;
  return ok ? OSCAR_OK : OSCAR_ERR_FILE;
}

extern "C" oscar_status oscar_rotation_file_info(const char* path, int32_t* n_layers, int32_t* n_kv_heads,
                                                  int32_t* d) {
  OSCAR_TRACE_CALL();
  if (!path || !n_layers || !n_kv_heads || !d) return OSCAR_ERR_INVALID_ARG;
  File in;
  in.f = std::fopen(path, "rb");
  if (!in.f) return OSCAR_ERR_FILE;
  char magic[8];
  uint32_t head[4];
  if (std::fread(magic, 1, 8, in.f) != 8 || std::memcmp(magic, kMagic, 8) != 0) return OSCAR_ERR_FILE;
  if (std::fread(head, 1, sizeof(head), in.f) != sizeof(head) || head[0] != kVersion) return OSCAR_ERR_FILE;
  if (!dims_ok(int32_t(head[1]), int32_t(head[2]), int32_t(head[3]))) return OSCAR_ERR_FILE;
  *n_layers = int32_t(head[1]);
  *n_kv_heads = int32_t(head[2]);
  *d = int32_t(head[3]);
  return OSCAR_OK;
}

extern "C" oscar_status oscar_rotation_file_read(const char* path, int32_t n_layers, int32_t n_kv_heads, int32_t d,
                                                  float* r_k, float* r_v, float* tau_k, float* tau_v) {
  OSCAR_TRACE_CALL();
  if (!path || !r_k || !r_v || !tau_k || !tau_v || !dims_ok(n_layers, n_kv_heads, d)) return OSCAR_ERR_INVALID_ARG;
  if (!little_endian()) return OSCAR_ERR_UNSUPPORTED;
  int32_t fl = 0, fh = 0, fd = 0;
  const oscar_status st = oscar_rotation_file_info(path, &fl, &fh, &fd);
  if (st != OSCAR_OK) return st;
  if (fl != n_layers || fh != n_kv_heads || fd != d) return OSCAR_ERR_INVALID_ARG;
  File in;
  in.f = std::fopen(path, "rb");
  if (!in.f) return OSCAR_ERR_FILE;
  // the whole file is checked before any output is written
  const size_t per = size_t(n_kv_heads) * d * d;
  const size_t body = 8 + 16 + size_t(n_layers) * (8 + 8 * per);
  std::vector<unsigned char> buf(body + 8);
  if (std::fread(buf.data(), 1, buf.size(), in.f) != buf.size()) return OSCAR_ERR_FILE;
  unsigned char extra;
  if (std::fread(&extra, 1, 1, in.f) != 0) return OSCAR_ERR_FILE;   // trailing bytes
  Fnv1a sum;
  sum.add(buf.data(), body);
  uint64_t h = 0;
  std::memcpy(&h, buf.data() + body, 8);
  if (h != sum.h) return OSCAR_ERR_FILE;
  const unsigned char* p = buf.data() + 24;
  for (int32_t l = 0; l < n_layers; ++l) {
    std::memcpy(tau_k + l, p, 4);
    std::memcpy(tau_v + l, p + 4, 4);
    std::memcpy(r_k + l * per, p + 8, per * 4);
    std::memcpy(r_v + l * per, p + 8 + per * 4, per * 4);
    p += 8 + 8 * per;
  }
  return OSCAR_OK;
}
