"""PIC link step on GB300 (binding is added with the C-ABI library)."""
