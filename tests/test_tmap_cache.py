"""CPU test of the TMA descriptor cache's key and eviction logic
(csrc/tmap_cache.h), compiled with g++ into a small driver: a hit returns
the stored descriptor; a change in any one field of the key (base address,
any extent, stride or box extent, data type, swizzle) misses; the least
recently used entry is the one evicted; a repeated insertion updates in place."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "exact_attention_forward_05_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "tmap_cache.h"
using namespace attn_internal;
struct Map { unsigned char bytes[128]; };
static TmapKey base_key() {
  TmapKey k; std::memset(&k, 0, sizeof(k));
  k.base = 0x7f0000001000ull;
  k.dims[0] = 128; k.dims[1] = 8192; k.dims[2] = 16; k.dims[3] = 2;
  k.strides[0] = 256; k.strides[1] = 256ull * 8192; k.strides[2] = 256ull * 8192 * 16;
  k.box[0] = 64; k.box[1] = 128; k.box[2] = 1; k.box[3] = 1;
  k.dtype = 9; k.swizzle = 3;
  return k;
}
static Map map_of(int tag) { Map m; std::memset(&m, tag, sizeof(m)); return m; }
#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)
int main() {
  TmapCache<Map, 4> c;
  Map out;
  TmapKey k = base_key();
  CHECK(!c.find(k, &out));
  c.insert(k, map_of(7));
  CHECK(c.find(k, &out) && out.bytes[0] == 7 && out.bytes[127] == 7);
  // every single-field change misses
  for (int f = 0; f < 14; ++f) {
    TmapKey m = base_key();
    switch (f) {
      case 0: m.base += 16; break;
      case 1: case 2: case 3: case 4: m.dims[f - 1] += 1; break;
      case 5: case 6: case 7: m.strides[f - 5] += 16; break;
      case 8: case 9: case 10: case 11: m.box[f - 8] += 1; break;
      case 12: m.dtype += 1; break;
      default: m.swizzle = 0; break;
    }
    CHECK(!c.find(m, &out));
  }
  // LRU: fill 4 slots, touch the first, insert a fifth -> the second is evicted
  c.clear();
  TmapKey ks[5];
  for (int i = 0; i < 5; ++i) { ks[i] = base_key(); ks[i].base += 4096ull * i; }
  for (int i = 0; i < 4; ++i) c.insert(ks[i], map_of(i + 1));
  CHECK(c.find(ks[0], &out) && out.bytes[0] == 1);
  c.insert(ks[4], map_of(5));
  CHECK(!c.find(ks[1], &out));
  CHECK(c.find(ks[0], &out) && out.bytes[0] == 1);
  CHECK(c.find(ks[2], &out) && out.bytes[0] == 3);
  CHECK(c.find(ks[3], &out) && out.bytes[0] == 4);
  CHECK(c.find(ks[4], &out) && out.bytes[0] == 5);
  // re-inserting a present key updates it in place (no second copy evicts anything)
  c.insert(ks[2], map_of(9));
  CHECK(c.find(ks[2], &out) && out.bytes[0] == 9);
  CHECK(c.find(ks[0], &out) && c.find(ks[3], &out) && c.find(ks[4], &out));
  std::printf("OK hits=%llu misses=%llu\n", (unsigned long long)c.hits(), (unsigned long long)c.misses());
  return 0;
}
"""


def test_tmap_cache_logic(tmp_path):
    gxx = "g++"
    src = tmp_path / "driver.cpp"
    exe = tmp_path / "driver"
    src.write_text(DRIVER)
    try:
        subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", f"-I{CSRC}", str(src), "-o", str(exe)],
                       check=True, capture_output=True, text=True)
    except FileNotFoundError:
        pytest.skip("g++ not available")
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr
