"""The whole path in float64: tables, append (encode + store), reconstruct, attend.

Ties the oracle modules together for one cache configuration.  Every step is
the plain definition or the pages' algorithm from the modules it calls; this
module only routes arrays (see ``codec``, ``layout``, ``attention``, ``headq``).
"""

import numpy as np

from . import attention, codebook, codec, layout, rotation, spectral, tables


class OracleContext:
    def __init__(self, head_dim, num_q_heads, num_kv_heads, batch, capacity,
                 k_codec, v_codec, seed, m=None, headq_rank=0, headq_bits=4, headq_basis=None,
                 spectral_k=None, spectral_v=None):
        """spectral_k / spectral_v: per KV head (E32, s32) storage-order tables of an SQU-KV side
        (oracle/spectral.py)."""
        d = head_dim
        self.d, self.Hq, self.Hkv, self.B, self.capacity = d, num_q_heads, num_kv_heads, batch, capacity
        self.G = num_q_heads // num_kv_heads
        self.k_codec, self.v_codec = k_codec, v_codec
        self.m = m or d
        self.seed = seed
        self.headq_rank, self.headq_bits = headq_rank, headq_bits
        self.C_K, self.T_K = codebook.fp32_tables(d, k_codec.bits)
        self.C_V, self.T_V = codebook.fp32_tables(d, v_codec.bits)
        self.D_K = tables.rotation_signs(seed, tables.STREAM_D_K, d) if k_codec.rotate else np.ones(d)
        self.D_V = tables.rotation_signs(seed, tables.STREAM_D_V, d) if v_codec.rotate else np.ones(d)
        self.R_K = rotation.rotation_matrix(self.D_K) if k_codec.rotate else np.eye(d)
        self.R_V = rotation.rotation_matrix(self.D_V) if v_codec.rotate else np.eye(d)
        self.S_K = tables.sketch_matrix(seed, tables.STREAM_S_K, self.m, d) if k_codec.qjl else None
        self.S_V = tables.sketch_matrix(seed, tables.STREAM_S_V, self.m, d) if v_codec.qjl else None
        self.U = None if headq_basis is None else np.asarray(headq_basis, dtype=np.float32)
        self.sq = {"k": spectral_k, "v": spectral_v}
        if k_codec.spectral or v_codec.spectral:
            self.C4, self.T4 = codebook.fp32_tables(d, spectral.TOP_BITS)
            self.C1, self.T1 = codebook.fp32_tables(d, spectral.FLOOR_BITS)
        self.shape = layout.CacheShape(batch, num_kv_heads, capacity, d, k_codec.bits, k_codec.qjl,
                                       v_codec.bits, v_codec.qjl, self.m, headq_rank, headq_bits,
                                       k_codec.spectral, v_codec.spectral)
        self.cache_bytes = layout.layout(self.shape)["total"]

    def new_cache(self):
        return np.zeros(self.cache_bytes, dtype=np.uint8)

    def encode_side(self, X, side, kvh=0):
        """Encode vectors X (N x d) of one KV head; returns the codec fields (+ side code for HeadQ K)."""
        cdc = self.k_codec if side == "k" else self.v_codec
        if cdc.spectral:
            E32, s32 = self.sq[side][kvh]
            return spectral.encode(X, side, E32, s32, self.C4, self.T4, self.C1, self.T1)
        if side == "k":
            f = codec.encode(X, self.k_codec, self.C_K, self.T_K, self.R_K, self.S_K)
            if self.headq_rank:
                f.update(codec.headq_encode(X, f["codes"], f["norm"], self.C_K, self.R_K,
                                            self.U[kvh].astype(np.float64), self.headq_bits))
            return f
        return codec.encode(X, self.v_codec, self.C_V, self.T_V, self.R_V, self.S_V)

    def packed_fields(self, f, side):
        cdc = self.k_codec if side == "k" else self.v_codec
        if cdc.spectral:
            return {side + "_codes": spectral.pack(f["codes"], side), side + "_norm": f["norm"]}
        bits = cdc.bits
        out = {side + "_codes": layout.pack_codes(f["codes"], bits), side + "_norm": f["norm"]}
        if "signs" in f:
            out[side + "_signs"] = layout.pack_stream(f["signs"].astype(np.int64), 1)
            out[side + "_rho"] = f["rho"]
        if side == "k" and self.headq_rank:
            out["k_side"] = layout.pack_side(f["side"])
            out["k_side_scale"] = f["side_scale"]
        return out

    def append(self, buf, K, V, start):
        """Encode K, V (B, H_kv, n_new, d) and store them at token start[b].. of each slab.

        Returns the per-slab field dicts {(b, h): (k_fields, v_fields)}.
        """
        K = np.asarray(K, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        n_new = K.shape[2]
        fields = {}
        for b in range(K.shape[0]):
            for h in range(K.shape[1]):
                fk = self.encode_side(K[b, h], "k", h)
                fv = self.encode_side(V[b, h], "v", h)
                layout.write_fields(buf, self.shape, b, h, int(start[b]), self.packed_fields(fk, "k"))
                layout.write_fields(buf, self.shape, b, h, int(start[b]), self.packed_fields(fv, "v"))
                fields[(b, h)] = (fk, fv)
        assert all(int(s) + n_new <= self.capacity for s in start)
        return fields

    def stored_fields(self, buf, side, b, h, T):
        """Parse the stored fields of tokens [0, T) of slab (b, h) back from the cache bytes."""
        bits = self.k_codec.bits if side == "k" else self.v_codec.bits
        cdc = self.k_codec if side == "k" else self.v_codec
        raw = layout.read_field(buf, self.shape, side + "_codes", b, h, 0, T)
        if cdc.spectral:
            return {"codes": spectral.unpack(raw, side, self.d),
                    "norm": layout.read_field(buf, self.shape, side + "_norm", b, h, 0, T, np.float32)}
        f = {"codes": layout.unpack_codes(raw, bits, self.d),
             "norm": layout.read_field(buf, self.shape, side + "_norm", b, h, 0, T, np.float32)}
        if cdc.qjl:
            f["signs"] = layout.unpack_stream(layout.read_field(buf, self.shape, side + "_signs", b, h, 0, T), 1, self.m) == 1
            f["rho"] = layout.read_field(buf, self.shape, side + "_rho", b, h, 0, T, np.float16)
        if side == "k" and self.headq_rank:
            f["side"] = layout.unpack_side(layout.read_field(buf, self.shape, "k_side", b, h, 0, T), self.headq_rank)
            f["side_scale"] = layout.read_field(buf, self.shape, "k_side_scale", b, h, 0, T, np.float16)
        return f

    def reconstruct(self, buf, b, h, T):
        """(K_hat, V_hat) of tokens [0, T) of slab (b, h), float64, from the stored bytes."""
        fk = self.stored_fields(buf, "k", b, h, T)
        fv = self.stored_fields(buf, "v", b, h, T)
        if self.k_codec.spectral and self.v_codec.spectral:
            Kh = spectral.reconstruct(fk["codes"], fk["norm"], "k", *self.sq["k"][h], self.C4, self.C1)
            Vh = spectral.reconstruct(fv["codes"], fv["norm"], "v", *self.sq["v"][h], self.C4, self.C1)
            return Kh, Vh
        Kh = codec.reconstruct(self.k_codec, fk["codes"], fk["norm"], self.C_K, self.R_K,
                               fk.get("rho"), fk.get("signs"), self.S_K,
                               fk.get("side"), fk.get("side_scale"),
                               None if self.U is None else self.U[h].astype(np.float64))
        Vh = codec.reconstruct(self.v_codec, fv["codes"], fv["norm"], self.C_V, self.R_V,
                               fv.get("rho"), fv.get("signs"), self.S_V)
        return Kh, Vh

    def decode(self, buf, q, seq_len, slabs=None):
        """Attention output (B, H_q, d) for queries q (B, H_q, d) over the stored cache.

        ``slabs`` limits the work to a list of (b, kv_head) pairs (others are left 0).
        """
        q = np.asarray(q, dtype=np.float64)
        out = np.zeros((self.B, self.Hq, self.d))
        todo = slabs if slabs is not None else [(b, h) for b in range(self.B) for h in range(self.Hkv)]
        for b, h in todo:
            T = int(seq_len[b])
            Kh, Vh = self.reconstruct(buf, b, h, T)
            for g in range(self.G):
                out[b, h * self.G + g] = attention.decode_attention(q[b, h * self.G + g], Kh, Vh)
        return out

    def logits(self, buf, q, seq_len, max_seq):
        """Scores q^T k_hat_j / sqrt(d) (B, H_q, max_seq), 0 beyond seq_len."""
        q = np.asarray(q, dtype=np.float64)
        out = np.zeros((self.B, self.Hq, max_seq))
        for b in range(self.B):
            T = int(seq_len[b])
            for h in range(self.Hkv):
                Kh, _ = self.reconstruct(buf, b, h, T)
                for g in range(self.G):
                    out[b, h * self.G + g, :T] = attention.logits(q[b, h * self.G + g], Kh)
        return out
