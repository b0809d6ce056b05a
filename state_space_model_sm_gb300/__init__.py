"""Mamba-2 SSD chunked selective scan for GB300 (sm_103a)."""
