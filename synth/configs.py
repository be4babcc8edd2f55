"""Workload definitions: shapes, dtypes, value distributions and seeds.

Each workload is a product-key memory lookup problem (Product-Key Memory,
"Factorising the key space"): B queries of H heads of width d_q, per-head
subkey tables [H, 2, n_keys, d_q/2], one shared value table
[n_keys**2, d_v], and a selection size k.  Variances below are the second
parameter of N(0, var).  This file holds sizes and distributions only.
"""

SEED_BASE = 0x504B4D00

# tensor ids of the counter-based streams (see gen.c)
TID_Q = 1
TID_KEYS = 2
TID_VALUES = 3
TID_MIX_MEAN = 4
TID_MIX_PICK = 5
TID_X = 6            # layer input of the query network
TID_QW = 7           # query network weight
TID_BN = 8           # BatchNorm gamma, beta, running mean, running var: 8, 9, 10, 11
TID_SEL = 12         # backward inputs: per-half subkey lists, picks, weights, dout: 12 .. 15

CONFIGS = {
    # fp32 everywhere; small enough for brute force over all n_keys**2 keys.
    "tiny": dict(cfg_id=0, B=64, H=1, d_q=64, n_keys=32, d_v=64, k=8, dtype="f32",
                 q_var=1.0, key_var=1.0, value_var=1.0 / 64, q_kind="normal"),
    # 64 MiB value table.
    "mid": dict(cfg_id=1, B=4096, H=4, d_q=512, n_keys=256, d_v=512, k=16, dtype="bf16",
                q_var=1.0, key_var=1.0 / 256, value_var=1.0 / 512, q_kind="normal"),
    # n_keys = 1024 (N = 2**20), k = 32, d = 1024: the page's worked sizes.
    "page": dict(cfg_id=2, B=16384, H=4, d_q=1024, n_keys=1024, d_v=1024, k=32, dtype="bf16",
                 q_var=1.0, key_var=1.0 / 512, value_var=1.0 / 1024, q_kind="normal"),
    # page shapes, 4x the queries, 8 heads, queries from a Zipf-weighted
    # 64-component Gaussian mixture (concentrated row usage).
    "skew": dict(cfg_id=3, B=65536, H=8, d_q=1024, n_keys=1024, d_v=1024, k=32, dtype="bf16",
                 q_var=1.0, key_var=1.0 / 512, value_var=1.0 / 1024, q_kind="mixture",
                 mix_components=64, mix_zipf_s=1.1, mix_sd=0.1),
    # the page workload's inputs (same seed), its value table kept as fp8 e4m3
    # codes with per-row scales (quantised from the bf16 table).
    "page_fp8": dict(cfg_id=2, B=16384, H=4, d_q=1024, n_keys=1024, d_v=1024, k=32,
                     dtype="bf16", value_format="fp8_e4m3", q_var=1.0, key_var=1.0 / 512,
                     value_var=1.0 / 1024, q_kind="normal"),
    # the whole layer on page shapes: layer input x [B, dim] -> query network
    # (Linear dim -> H*d_q, BatchNorm with running statistics) -> lookup -> read.
    # x ~ N(0, 1), W ~ N(0, 1/dim), so the queries are about N(0, 1) as in page.
    "page_layer": dict(cfg_id=2, B=16384, H=4, d_q=1024, n_keys=1024, d_v=1024, k=32,
                       dtype="bf16", q_var=1.0, key_var=1.0 / 512, value_var=1.0 / 1024,
                       q_kind="normal", qnet_dim=1024, bn_eps=1e-5),
    # a training step on page shapes: the forward pass, then the backward
    # pass for its selection with a seeded output gradient dout ~ N(0, 1)
    # (dq; dsubkeys and dvalues accumulated in fp32).
    "page_train": dict(cfg_id=2, B=16384, H=4, d_q=1024, n_keys=1024, d_v=1024, k=32,
                       dtype="bf16", q_var=1.0, key_var=1.0 / 512, value_var=1.0 / 1024,
                       q_kind="normal", train=True),
    # the same training step with the value-table gradient in sparse form
    # (distinct selected rows and their gradient rows) instead of added to a
    # dense fp32 table.
    "page_train_sparse": dict(cfg_id=2, B=16384, H=4, d_q=1024, n_keys=1024, d_v=1024, k=32,
                              dtype="bf16", q_var=1.0, key_var=1.0 / 512, value_var=1.0 / 1024,
                              q_kind="normal", train=True, sparse_grad=True),
    # the mid workload's inputs (same seed) searched flat: every query scored
    # against all N = n_keys^2 materialised full keys (the search the
    # factorisation replaces), then the same value read.
    "mid_flat": dict(cfg_id=1, B=4096, H=4, d_q=512, n_keys=256, d_v=512, k=16, dtype="bf16",
                     q_var=1.0, key_var=1.0 / 256, value_var=1.0 / 512, q_kind="normal",
                     flat=True),
    # 16 GiB value table.
    "large": dict(cfg_id=4, B=32768, H=4, d_q=2048, n_keys=2048, d_v=2048, k=32, dtype="bf16",
                  q_var=1.0, key_var=1.0 / 1024, value_var=1.0 / 2048, q_kind="normal"),
}


def seed_of(cfg):
    return SEED_BASE + cfg["cfg_id"]


def n_rows(cfg):
    return cfg["n_keys"] ** 2
