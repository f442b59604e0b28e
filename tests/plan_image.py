"""Reader of the plan image (layout documented in csrc/pka_plan_image.h)."""
import numpy as np

HEADER = ["magic", "total_words", "num_decode_ctas", "num_decode_items", "num_prefill_ctas",
          "num_prefill_items", "num_merge_tasks", "num_partial_records", "off_decode_cta_ptr",
          "off_decode_items", "off_prefill_cta_ptr", "off_prefill_items", "off_merge_tasks",
          "decode_heads_per_cta", "graph_mode", "off_merge_slots", "num_decode_joins",
          "off_decode_joins", "num_dequant_units", "off_dequant_units", "dequant_rows"]
ITEM = ["req", "kv_head0", "n_kv_heads", "q_row0", "q_local0", "q_count", "qo_len", "kv_len",
        "kv_base", "t0", "t1", "out_rec", "mask_lo", "mask_hi", "flags", "join"]
MERGE = ["out_row", "head", "rec_first", "nslots", "rec_stride"]
JOIN = ["arrived", "rec_first", "nslots", "rec_stride"]
DEQUANT = ["kv_base", "kv_len", "dst_row0"]


def parse(buf: np.ndarray):
    w = np.frombuffer(buf.tobytes(), dtype=np.int32)
    h = {k: int(w[i]) for i, k in enumerate(HEADER)}
    assert h["magic"] == 0x31414B50

    def items(off, n):
        return [dict(zip(ITEM, map(int, w[off + 16 * i: off + 16 * (i + 1)]))) for i in range(n)]

    dec_ptr = w[h["off_decode_cta_ptr"]: h["off_decode_cta_ptr"] + h["num_decode_ctas"] + 1]
    pre_ptr = w[h["off_prefill_cta_ptr"]: h["off_prefill_cta_ptr"] + h["num_prefill_ctas"] + 1]
    merges = [dict(zip(MERGE, map(int, w[h["off_merge_tasks"] + 8 * i:
                                          h["off_merge_tasks"] + 8 * i + 5])))
              for i in range(h["num_merge_tasks"])]
    joins = []
    if h["off_decode_joins"]:
        o = h["off_decode_joins"]
        joins = [dict(zip(JOIN, map(int, w[o + 4 * i: o + 4 * (i + 1)])))
                 for i in range(h["num_decode_joins"])]
    slots = []
    if h["off_merge_slots"]:
        o = h["off_merge_slots"]
        slots = [int(x) for x in w[o:o + h["num_partial_records"]]]
    dequant = []
    if h["off_dequant_units"]:
        o = h["off_dequant_units"]
        dequant = [dict(zip(DEQUANT, map(int, w[o + 4 * i: o + 4 * i + 3])))
                   for i in range(h["num_dequant_units"])]
    return {"header": h, "decode_cta_ptr": [int(x) for x in dec_ptr], "merge_slots": slots,
            "dequant_units": dequant,
            "decode_items": items(h["off_decode_items"], h["num_decode_items"]),
            "prefill_cta_ptr": [int(x) for x in pre_ptr],
            "prefill_items": items(h["off_prefill_items"], h["num_prefill_items"]),
            "merges": merges, "joins": joins}
