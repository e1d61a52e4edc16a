"""Pins for the storage arithmetic: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV
quantization", description, storage paragraph (K+V bytes per token per KV head at head_dim 256,
and the whole-cache GiB for 262,144 tokens x 16 layers x 4 KV heads)."""
import json

from oracle import storage
from conftest import golden_path


def test_bytes_per_token_per_kv_head():
    g = json.load(open(golden_path("storage.json")))
    for bits, b in g["kv_bytes_per_token_per_kv_head"].items():
        assert storage.kv_bytes_per_token_head(g["head_dim"], int(bits)) == b


def test_full_cache_gib():
    g = json.load(open(golden_path("storage.json")))
    fc = g["full_cache"]
    exact = {16: 17_179_869_184, 8: 8_657_043_456, 6: 6_509_559_808, 4: 4_362_076_160}
    for bits, gib in g["full_cache_gib_printed"].items():
        n = storage.cache_bytes(fc["tokens"], fc["layers"], fc["kv_heads"], g["head_dim"],
                                int(bits))
        assert n == exact[int(bits)]
        assert abs(n / 2 ** 30 - gib) <= g["printed_precision_gib"]
